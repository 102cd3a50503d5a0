// gemm_tf32.cu - instantiation and launch of the tcgen05 implicit-GEMM kernels
// for fp32 operands (3xTF32).
#include "kernels.h"

namespace c2d {

cudaError_t launch_conv_gemm_tf32(const ConvGemmParams& p, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(conv_gemm_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  launch_k(conv_gemm_kernel<0, false>, grid, kThreads, smem, st, 1, p);
  return cudaGetLastError();
}

cudaError_t launch_wgrad_gemm_tf32(const WgradParams& p, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(wgrad_gemm_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  launch_k(wgrad_gemm_kernel<0, false>, grid, kThreads, smem, st, 1, p);
  return cudaGetLastError();
}

}  // namespace c2d
