// gemm_bf16.cu - instantiation and launch of the tcgen05 implicit-GEMM kernels
// for bf16 operands.
#include "kernels.h"

namespace c2d {

cudaError_t launch_conv_gemm_bf16(const ConvGemmParams& p, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(conv_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  conv_gemm_kernel<1><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wgrad_gemm_bf16(const WgradParams& p, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(wgrad_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  wgrad_gemm_kernel<1><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace c2d
