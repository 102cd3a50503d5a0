// gemm_bf16.cu - instantiation and launch of the tcgen05 implicit-GEMM kernels
// for bf16 operands.
#include "kernels.h"

namespace c2d {

// One instantiation of the bf16 fprop / dgrad kernel (see conv_gemm_kernel's PAIR and BMN).
template <bool PAIR, bool BMN>
static cudaError_t launch_conv(const ConvGemmParams& p, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(conv_gemm_kernel<1, PAIR, BMN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (PAIR) return launch_k(conv_gemm_kernel<1, PAIR, BMN>, grid, kThreads, smem, st, 2, p);  // clusters of two
  launch_k(conv_gemm_kernel<1, PAIR, BMN>, grid, kThreads, smem, st, 1, p);
  return cudaGetLastError();
}

cudaError_t launch_conv_gemm_bf16(const ConvGemmParams& p, int grid, size_t smem, cudaStream_t st) {
  if (p.b_mn) return p.pair ? launch_conv<true, true>(p, grid, smem, st) : launch_conv<false, true>(p, grid, smem, st);
  return p.pair ? launch_conv<true, false>(p, grid, smem, st) : launch_conv<false, false>(p, grid, smem, st);
}

int conv_gemm_pair_clusters(size_t smem) {
  if (cudaFuncSetAttribute(conv_gemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, conv_gemm_kernel<1, true>, &cfg) != cudaSuccess) return 0;
  return n;
}

// Launch configuration of a kernel run in clusters of two CTAs.
static cudaLaunchConfig_t pair_config(int grid, size_t smem, cudaStream_t st, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t launch_wgrad_gemm_bf16(const WgradParams& p, int grid, size_t smem, cudaStream_t st) {
  if (!p.pair) {
    cudaError_t e = cudaFuncSetAttribute(wgrad_gemm_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    launch_k(wgrad_gemm_kernel<1, false>, grid, kThreads, smem, st, 1, p);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(wgrad_gemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(wgrad_gemm_kernel<1, true>, grid, kThreads, smem, st, 2, p);
}

int wgrad_gemm_pair_clusters(size_t smem) {
  if (cudaFuncSetAttribute(wgrad_gemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  cudaLaunchAttribute at[1];
  const cudaLaunchConfig_t cfg = pair_config(2, smem, nullptr, at);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, wgrad_gemm_kernel<1, true>, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace c2d
