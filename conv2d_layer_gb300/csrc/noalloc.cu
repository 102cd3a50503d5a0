// noalloc.cu - conv2d_fwd_train for callers that cannot allocate device
// memory.
//
// Who needs it: a caller whose device memory is fixed once at start-up and
// who may not allocate afterwards (a deployment with a locked memory budget,
// a control or training loop that must not stall: cudaMalloc / cudaFree can
// synchronise the device), or a caller that only receives the tensors it
// passes in and has no way to obtain a scratch buffer of its own. Such a
// caller cannot hand conv2d_fwd_train the workspace it asks for.
//
// What it does: the same launches as conv2d_fwd_train, with the workspace
// replaced by a file-scope device array of kStaticScratchBytes. Every GPU that
// loads the library holds that array until the process exits. Its device
// address is looked up once per device (cudaGetSymbolAddress, with that device
// current) on the first call made on the device; in host code the array's
// name is only a host-side handle and is never passed to a kernel.
#include <cuda_runtime.h>

#include <mutex>

#include "conv2d.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

}  // namespace

extern "C" int conv2d_fwd_train_noalloc(const conv2d_desc* desc, const void* x, const void* w, const float* bias,
                                        const float* gamma, const float* beta, float* running_mean,
                                        float* running_var, void* pre_act, float* save_mean, float* save_inv_std,
                                        void* y, void* stream) {
  const int rc = conv2d_validate(desc);
  if (rc != CONV2D_OK) return rc;
  // sizes beyond the static array are refused before anything is launched
  if (conv2d_workspace_size(desc, CONV2D_OP_FWD_TRAIN) > kStaticScratchBytes) return CONV2D_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CONV2D_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return CONV2D_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  // The forward pass overwrites every scratch byte it later reads (per-tile
  // statistics, packed operands), so nothing needs clearing between calls.
  return conv2d_fwd_train(desc, x, w, bias, gamma, beta, running_mean, running_var, pre_act, save_mean,
                          save_inv_std, y, scratch, kStaticScratchBytes, stream);
}
