// kernels_cg1.cu -- single-CTA (cta_group::1) instances of the fused GEMM kernel.
#include "gemm_kernel.cuh"
#include "launch.h"

namespace ge {

template <int BN>
static cudaError_t launch_one(const KParams &p, int grid, int smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<1, BN>, p);
}

cudaError_t gemm_prepare_cg1(int bn, int smem) {
  switch (bn) {
    case 64: return cudaFuncSetAttribute(gemm_epi_kernel<1, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 128: return cudaFuncSetAttribute(gemm_epi_kernel<1, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 256: return cudaFuncSetAttribute(gemm_epi_kernel<1, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_launch_cg1(int bn, const KParams &p, int grid, int smem, cudaStream_t s) {
  switch (bn) {
    case 64: return launch_one<64>(p, grid, smem, s);
    case 128: return launch_one<128>(p, grid, smem, s);
    case 256: return launch_one<256>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ge
