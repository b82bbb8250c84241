// kernels_cg2.cu -- CTA-pair (cta_group::2, 2x1 cluster) instances of the fused GEMM kernel.
#include "gemm_kernel.cuh"
#include "launch.h"

namespace ge {

template <int BN>
static cudaLaunchConfig_t make_cfg(int grid, int smem, cudaStream_t s, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int BN>
static cudaError_t launch_one(const KParams &p, int grid, int smem, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg<BN>(grid, smem, s, attr);
  return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<2, BN>, p);
}

template <int BN>
static cudaError_t clusters_one(int smem, int *n) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg<BN>(2, smem, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(n, gemm_epi_kernel<2, BN>, &cfg);
}

cudaError_t gemm_prepare_cg2(int bn, int smem) {
  switch (bn) {
    case 128: return cudaFuncSetAttribute(gemm_epi_kernel<2, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 256: return cudaFuncSetAttribute(gemm_epi_kernel<2, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_launch_cg2(int bn, const KParams &p, int grid, int smem, cudaStream_t s) {
  switch (bn) {
    case 128: return launch_one<128>(p, grid, smem, s);
    case 256: return launch_one<256>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_max_active_clusters_cg2(int bn, int smem, int *n) {
  switch (bn) {
    case 128: return clusters_one<128>(smem, n);
    case 256: return clusters_one<256>(smem, n);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ge
