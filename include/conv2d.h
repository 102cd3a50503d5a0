/*
 * conv2d.h - C ABI of the GB300 (sm_103a) conv2d training-step library
 * (libconv2d.so).
 *
 * One NHWC 2D convolution layer: conv + bias, optional training-mode batch
 * norm, layer norm or group norm, activation; and its backward pass. The operation is the one defined by
 * the rl-tools conv2d layer pages ("operations_generic.h": `forward`,
 * `evaluate`, `backward`, `backward_input`, `backward_full`; the CUDA page
 * "operations_cuda.h" splits the same work into cuDNN calls and per-channel
 * kernels). The layer spec (N,H,W,IC,OC,KH,KW,stride,pad, normalization,
 * activation, eps, momentum, type policy) follows the template parameters
 * those pages read from their LayerSpec.
 *
 * Conventions (all calls):
 *   - Tensors are dense, contiguous NHWC: x [N][H][W][IC], y / pre_act / dy
 *     [N][OH][OW][OC], weights w [OC][KH][KW][IC]; OH = (H+2*pad-KH)/stride+1
 *     (floor), OW likewise; symmetric zero padding; cross-correlation (no
 *     kernel flip); no dilation, no groups.
 *   - x, w, pre_act, y, dy, dx have the element type named by desc->dtype
 *     (CONV2D_FP32: float; CONV2D_BF16: bfloat16). bias, gamma, beta, running
 *     statistics, saved statistics and every parameter gradient are float32.
 *   - Every pointer is a DEVICE pointer on the current CUDA device, aligned to
 *     16 bytes. The caller owns every buffer; the library allocates no device
 *     memory on any path. Scratch space is the caller's workspace `ws` of at
 *     least conv2d_workspace_size(desc, op) bytes (alignment 256 bytes); its
 *     contents need not be initialised and are clobbered.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Buffers must not be touched by other work until the
 *     stream reaches the call. Calls that share a workspace must be ordered.
 *   - Return value: CONV2D_OK, or an error code from host-side validation or
 *     launch (no kernel is launched when validation fails). Device-side
 *     failures (a bounded wait that ran out) are reported later by
 *     conv2d_device_status().
 *   - Accumulate / overwrite semantics follow `backward_full`: dw, dbias,
 *     dgamma, dbeta are ACCUMULATED into (the caller zeroes them, as the
 *     pages' `zero_gradient` does); dx is OVERWRITTEN.
 *   - The library is stateless apart from per-device constant data; it is
 *     safe to call from several host threads.
 *   - Per-device data is looked up once, on the first call made on a device,
 *     and cached for the life of the process: the SM count, the device
 *     address of the library's error word and of the static scratch array of
 *     conv2d_fwd_train_noalloc. cudaDeviceReset() on a device invalidates
 *     those addresses, so resetting a device while this library is loaded in
 *     the process is not supported.
 */
#ifndef CONV2D_GB300_H
#define CONV2D_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    CONV2D_OK = 0,
    CONV2D_ERR_INVALID_ARG = 1, /* bad size, NULL or misaligned pointer, bad enum, eps<=0, momentum outside [0,1] */
    CONV2D_ERR_UNSUPPORTED = 2, /* valid but not implemented (stride > 8, sizes beyond 2^31 elements) */
    CONV2D_ERR_WORKSPACE = 3,   /* ws NULL or smaller than conv2d_workspace_size() */
    CONV2D_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed (launch, tensor-map encode) */
    CONV2D_ERR_TIMEOUT = 5      /* a device-side bounded wait expired (reported by conv2d_device_status) */
};

/* Normalization (the pages' `Normalization` enum, plus the group norm of the
 * WebGPU page's GroupNorm backward). BATCH: per-channel statistics over
 * N*OH*OW with running statistics. LAYER: per-image statistics over OH*OW*OC
 * of the stored pre-activations (the pages' LAYER_NORM branches), per-channel
 * gamma / beta, no running statistics. GROUP: desc.groups groups of OC/groups
 * consecutive channels, statistics per (image, group) over OH*OW*OC/groups
 * stored pre-activations, per-channel gamma / beta, no running statistics
 * (GROUP with groups = 1 computes LAYER). */
enum { CONV2D_NORM_NONE = 0, CONV2D_NORM_BATCH = 1, CONV2D_NORM_LAYER = 2, CONV2D_NORM_GROUP = 3 };

/* Activation applied after (optional) normalization. */
enum { CONV2D_ACT_IDENTITY = 0, CONV2D_ACT_RELU = 1, CONV2D_ACT_TANH = 2, CONV2D_ACT_SIGMOID = 3 };

/* Element type of x, w, pre_act, y, dy, dx. FP32 runs the contractions as
 * 3xTF32 (split operands, fp32 accumulation) for fp32 accuracy; BF16 runs
 * bf16 x bf16 -> fp32 accumulation. */
enum { CONV2D_FP32 = 0, CONV2D_BF16 = 1 };

/* Operation selector for conv2d_workspace_size(). */
enum { CONV2D_OP_FWD_TRAIN = 0, CONV2D_OP_FWD_INFER = 1, CONV2D_OP_BWD = 2 };

/* Layer spec. eps is read for BATCH and LAYER norm (1/sqrt(var+eps), biased
 * variance); momentum only for BATCH
 * (running = (1-momentum)*running + momentum*batch, biased batch variance).
 * bn_eval != 0 selects batch norm in evaluation mode inside training (the
 * pages' mode::Evaluation): conv2d_fwd_train normalises with the running
 * statistics, writes them as save_mean / save_inv_std (= 1/sqrt(var+eps)) and
 * updates nothing; conv2d_bwd then uses the frozen-statistics backward
 * (d_conv = act'(bn) * dy * gamma * inv_std). Zero keeps training mode.
 * Layer and group norm have no evaluation mode on the pages: bn_eval is
 * ignored there. groups is read only for GROUP norm (1 <= groups, OC % groups
 * == 0). */
typedef struct {
    int32_t N, H, W, IC, OC, KH, KW, stride, pad;
    int32_t norm, act, dtype;
    float eps, momentum;
    int32_t bn_eval;
    int32_t groups;
} conv2d_desc;

/* Output spatial size. Returns CONV2D_OK or CONV2D_ERR_INVALID_ARG. */
int conv2d_out_hw(const conv2d_desc* desc, int32_t* OH, int32_t* OW);

/* Host-side validation of a layer spec alone (no pointers). */
int conv2d_validate(const conv2d_desc* desc);

/* Bytes of workspace needed by `op` for this spec (0 if the spec is invalid). */
size_t conv2d_workspace_size(const conv2d_desc* desc, int op);

/* Training forward (`forward` on the generic page; cuDNN conv + bias, batch
 * statistics, affine and activation kernels on the CUDA page).
 *   pre_act  [N][OH][OW][OC] out: conv + bias (the pages' `pre_activations`)
 *   y        [N][OH][OW][OC] out: activation(normalised pre_act)
 *   BATCH norm (else may be NULL):
 *     gamma, beta [OC] in; running_mean, running_var [OC] in/out (EMA update);
 *     save_mean, save_inv_std [OC] out: batch mean and 1/sqrt(var+eps) that
 *     conv2d_bwd needs.
 *   LAYER norm: gamma, beta [OC] in; save_mean, save_inv_std [N] out: the
 *     per-image mean and 1/sqrt(var+eps) of the stored pre_act;
 *     running_mean / running_var are not read and may be NULL.
 *   GROUP norm: as LAYER with save_mean, save_inv_std [N*groups] (index
 *     n*groups + g).
 *   bias may be NULL (treated as zero). */
int conv2d_fwd_train(const conv2d_desc* desc, const void* x, const void* w, const float* bias,
                     const float* gamma, const float* beta, float* running_mean, float* running_var,
                     void* pre_act, float* save_mean, float* save_inv_std, void* y,
                     void* ws, size_t ws_bytes, void* stream);

/* Training forward without a caller workspace. The pages have no counterpart
 * of this call; it exists for callers that cannot allocate device memory: a
 * process whose device memory is fixed at start-up and that may not allocate
 * afterwards (cudaMalloc / cudaFree can synchronise the device and can fail
 * mid-run), or code that is handed only the tensors it passes here and has
 * no way to obtain a scratch buffer.
 * Same arguments and results as conv2d_fwd_train minus ws / ws_bytes. Its
 * scratch is one static 32 MiB device array inside the library (every GPU
 * that loads the library holds it until the process exits). A spec whose
 * conv2d_workspace_size(desc, CONV2D_OP_FWD_TRAIN) exceeds 32 MiB is refused
 * with CONV2D_ERR_WORKSPACE before anything is launched. The first call on a
 * device looks up the array's device address (with that device current);
 * make that first call before any stream capture. All calls share the array
 * and a call rewrites every scratch byte it reads, so nothing is cleared
 * between calls, but calls that overlap on the GPU (several streams, several
 * host threads) race on it: order them. */
int conv2d_fwd_train_noalloc(const conv2d_desc* desc, const void* x, const void* w, const float* bias,
                             const float* gamma, const float* beta, float* running_mean, float* running_var,
                             void* pre_act, float* save_mean, float* save_inv_std, void* y, void* stream);

/* Inference forward (`evaluate`): y = act(norm(conv + bias)), batch norm with
 * the running statistics (`bn_stats_eval` / `bn_forward_eval_running` on the
 * CUDA page), layer / group norm with per-image (per-group) statistics of the
 * stored conv output computed on the fly; no state is written. gamma, beta
 * are read for BATCH, LAYER and GROUP norm, running_mean, running_var only
 * for BATCH. */
int conv2d_fwd_infer(const conv2d_desc* desc, const void* x, const void* w, const float* bias,
                     const float* gamma, const float* beta, const float* running_mean,
                     const float* running_var, void* y, void* ws, size_t ws_bytes, void* stream);

/* Backward (`backward_full`; `backward_input` when dw..dbeta are all NULL;
 * `backward` when dx is NULL). Inputs: x, w, pre_act and (BATCH / LAYER /
 * GROUP) gamma, beta, save_mean, save_inv_std from conv2d_fwd_train,
 * dy = dLoss/dy.
 *   dx [N][H][W][IC]   out (overwritten), may be NULL
 *   dw [OC][KH][KW][IC], dbias [OC]        accumulated, may be NULL together
 *   dgamma, dbeta [OC] (with a norm)        accumulated, may be NULL together
 * The norm backward uses the saved statistics, not recomputed ones; under
 * layer / group norm its projection sums run over each image (group): the
 * GroupNorm backward of the WebGPU page ("groupnorm_backward.wgsl") with the
 * activation derivative in front and the dgamma / dbeta it leaves out.
 * At least one of dx / dw must be non-NULL. */
int conv2d_bwd(const conv2d_desc* desc, const void* x, const void* w, const float* gamma,
               const float* beta, const void* pre_act, const float* save_mean,
               const float* save_inv_std, const void* dy, void* dx, float* dw, float* dbias,
               float* dgamma, float* dbeta, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, then reads and clears this device's error word,
 * which kernels set when a bounded wait expires. Returns CONV2D_OK,
 * CONV2D_ERR_TIMEOUT (with *site, if non-NULL, set to the wait site code) or
 * CONV2D_ERR_CUDA. */
int conv2d_device_status(void* stream, int32_t* site);

/* Diagnostic for the device-side failure path (no counterpart on the pages).
 * Launches one block whose thread waits, with the library's bounded wait, on a
 * barrier that nothing completes. After the wait limit (about 2 s) the wait
 * gives up, records site 6 in the device error word and the kernel ends; no
 * fault, trap or hang is involved and the context stays usable.
 * conv2d_device_status then returns CONV2D_ERR_TIMEOUT with site 6. */
int conv2d_selftest_wait_limit(void* stream);

/* Human-readable name of a status code (static string). */
const char* conv2d_status_str(int status);

/* Kernel timing for measurement. While enabled (on != 0), every kernel the
 * library launches is bracketed by CUDA events on its stream and recorded in
 * a fixed ring of 256 launches. conv2d_prof_read synchronises the device and
 * copies up to `cap` records (oldest first): a static kernel name and the
 * elapsed milliseconds; it returns the number copied and clears the ring.
 * Off by default; when off no events are recorded. */
int conv2d_prof_enable(int on);
int conv2d_prof_read(const char** names, float* ms, int cap);

#ifdef __cplusplus
}
#endif
#endif /* CONV2D_GB300_H */
