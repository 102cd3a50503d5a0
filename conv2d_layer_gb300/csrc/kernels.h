// kernels.h - launchers shared between the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include "conv_gemm.cuh"

namespace c2d {

// Launch with programmatic stream serialization (see pdl_entry, which every kernel runs first) and,
// for cluster > 1, thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// tcgen05 GEMMs (gemm_bf16.cu / gemm_tf32.cu)
cudaError_t launch_conv_gemm_bf16(const ConvGemmParams& p, int grid, size_t smem, cudaStream_t st);
// Clusters of two CTAs of the pair form that can be resident at once (0 if the query fails).
int conv_gemm_pair_clusters(size_t smem);
cudaError_t launch_conv_gemm_tf32(const ConvGemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_wgrad_gemm_bf16(const WgradParams& p, int grid, size_t smem, cudaStream_t st);
int wgrad_gemm_pair_clusters(size_t smem);
cudaError_t launch_wgrad_gemm_tf32(const WgradParams& p, int grid, size_t smem, cudaStream_t st);

// Per-phase description of the dgrad weight matrix (see prep_dgrad_weights).
struct DgradWeightTable {
  int n;
  int flip;  // columns in reversed tap order within each phase (for TMA im2col, whose offsets are >= 0)
  int col_off[kMaxPhases];
  int Th[kMaxPhases], Tw[kMaxPhases], rh[kMaxPhases], rw[kMaxPhases];
};

// Row walk of an NHWC tensor seen as [rows][C]: G blocks, each owning a
// contiguous slice of rows. The rows form `segs` segments of seg_rows rows
// (1 segment for batch norm and no norm; one per image for layer norm), each
// split over bps blocks, so that no block straddles a segment and the
// per-block partials of one segment are contiguous (block = seg * bps + j).
struct RowWalk {
  long rows;
  int C;
  int G;
  long rows_per_block;
  int segs, bps;
  long seg_rows;
  int cpg;     // statistics per channel (0, batch norm) or per image and group of cpg channels
  int stream;  // rows move through shared memory by bulk TMA copies (vector path)
  int R;       // rows per streamed chunk
  int* err;    // device error word for bounded waits
};
RowWalk make_walk(long rows, int C, int dtype, int sms, int segs, int cpg, int per_sm = 2);

// elementwise / reduction kernels (bn_kernels.cu); dtype 0 = fp32, 1 = bf16
cudaError_t launch_pack_channels(int dtype, const void* src, void* dst, long rows, int C, int Cp, cudaStream_t st);
cudaError_t launch_prep_fprop_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int taps, int IC,
                                      int ICp, cudaStream_t st);
cudaError_t launch_prep_dgrad_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int KH, int KW,
                                      int IC, int ICp, int OCp, int S, int Kd, const DgradWeightTable& t,
                                      cudaStream_t st);
// Phase-merged dgrad weights B[(ph_h, ph_w, icp)][(tap, oc)] (see prep_dgrad_merged_weights_kernel).
cudaError_t launch_prep_dgrad_merged_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int KH, int KW,
                                             int IC, int ICp, int OCp, int S, cudaStream_t st);
cudaError_t launch_bn_stats_finalize(const float* part, const RowWalk& wk, float eps, float momentum, float* mean,
                                     float* inv_std, float* rm, float* rv, cudaStream_t st);
// rev != 0 walks the rows last to first (streamed path): the kernel starts on the rows the previous
// kernel touched last, which are still in L2.
cudaError_t launch_bn_apply(int dtype, const void* pre, void* y, const RowWalk& wk, const float* mean,
                            const float* inv_std, const float* gamma, const float* beta, int act, int rev,
                            cudaStream_t st);
// part[G][C][nv]: (sum d_norm, sum d_norm z) and, with nv = 3 (streamed batch-norm walks only), sum (x - mean)
cudaError_t launch_bn_bwd_reduce(int dtype, const void* pre, const void* dy, const RowWalk& wk, const float* mean,
                                 const float* inv_std, const float* gamma, const float* beta, int act, float* part,
                                 int nv, cudaStream_t st);
// sums[c][v] over the G block partials (v < nv); mode 0: c12 <- sums, dbeta += s0, dgamma += s1;
// mode 1: dbias += s0.
cudaError_t launch_sum_finalize(const float* part, const RowWalk& wk, int nv, int mode, float* c12, float* acc0,
                                float* acc1, cudaStream_t st);
// Batch norm with d_conv formed inside the GEMM producers: from the nv = 3 reduce partials, c12, dbeta,
// dgamma, dbias (each accumulated where non-null) and the per-channel terms tbl[4][C] of d_conv
// (G, B', Q, S': t = G x + B', d_conv = G d_norm + Q x + S').
cudaError_t launch_bn_bwd_fused_finalize(const float* part, const RowWalk& wk, const float* mean,
                                         const float* inv_std, const float* gamma, const float* beta, float* c12,
                                         float* dbeta, float* dgamma, float* dbias, float* tbl, cudaStream_t st);
// d_conv under batch norm (c12 = per-channel sums from launch_sum_finalize; null: evaluation mode) or,
// on a segmented walk, layer norm (c12 + 2C = the per-image sums of launch_ln_seg_finalize).
cudaError_t launch_bn_bwd_apply(int dtype, const void* pre, const void* dy, const RowWalk& wk, int Cp,
                                const float* mean, const float* inv_std, const float* gamma, const float* beta,
                                int act, const float* c12, void* dconv, float* part, cudaStream_t st);
cudaError_t launch_act_bwd(int dtype, const void* pre, const void* dy, const RowWalk& wk, int Cp, int act,
                           void* dconv, float* part, cudaStream_t st);
// Layer norm: per-image mean / inv_std from the fprop epilogue's per-pixel (mean, M2) partials
// [n_images * hw][n_tiles][halves][2] (half 0 = the first hcols columns of a tile).
cudaError_t launch_ln_stats_finalize(const float* rstats, int n_images, long hw, int n_tiles, int halves, int BN,
                                     int hcols, int OC, float eps, float* mean, float* inv_std, cudaStream_t st);
// Layer / group norm backward: per-(image, group) sums of gamma * d_norm and gamma * d_norm * z from the
// bwd-reduce partials of an image-aligned walk, written to out[2s], out[2s + 1] (s = image * groups + g).
cudaError_t launch_norm_seg_finalize(const float* part, const RowWalk& wk, const float* gamma, float* out,
                                     cudaStream_t st);
// Group norm forward statistics: per-block, per-channel (rows, mean, M2) of the stored pre-activations on
// an image-aligned walk, then their per-(image, group) merge.
cudaError_t launch_norm_stats(int dtype, const void* pre, const RowWalk& wk, int rev, float* part,
                              cudaStream_t st);
cudaError_t launch_gn_stats_finalize(const float* part, const RowWalk& wk, float eps, float* mean, float* inv_std,
                                     cudaStream_t st);
// Column-form dgrad for small input-channel counts with stride: dcol = d_conv x B (a 1x1 fprop over
// d_conv with B[(tap, icp)][oc] from prep_col2im_weights), then dX gathered from dcol per element.
cudaError_t launch_prep_col2im_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int taps, int IC,
                                       int ICp, int OCp, cudaStream_t st);
cudaError_t launch_col2im(int dtype, const void* dcol, void* dx, int N, int H, int W, int IC, int ICp, int OH, int OW,
                          int KH, int KW, int S, int P, cudaStream_t st);
// dW += the sum of the split partials; with dbias, also dbias[c] += the sum of bpart[0..bG)[c] (the dbias
// finalize, in OC more blocks of the same launch).
cudaError_t launch_wgrad_reduce(const float* partial, int splits, int OC, int taps, int ICp, int IC, float* dw,
                                const float* bpart, int bG, float* dbias, cudaStream_t st);
cudaError_t launch_bn_eval_stats(const float* rm, const float* rv, float eps, int C, float* mean, float* inv_std,
                                 cudaStream_t st);
cudaError_t launch_infer_fold(const float* bias, const float* gamma, const float* beta, const float* rm,
                              const float* rv, float eps, int norm, int OC, float* scale, float* shift,
                              cudaStream_t st);

}  // namespace c2d
