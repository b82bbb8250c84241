// launch.h -- host-side entry points of the kernel translation units.
#pragma once

#include <cuda_runtime_api.h>

#include "common.cuh"

namespace ge {

// GEMM + fused epilogue kernel, instantiated for (cta_group, BN) in
// {(1, 64), (1, 128), (1, 256), (2, 128), (2, 256)}.
bool gemm_variant_exists(int cg, int bn);
cudaError_t gemm_prepare(int cg, int bn, int smem_bytes);  // opt in to the dynamic smem size
cudaError_t gemm_launch(int cg, int bn, const KParams &p, int grid, int smem_bytes,
                        cudaStream_t stream);
cudaError_t gemm_max_active_clusters(int cg, int bn, int smem_bytes, int *clusters);

// per-translation-unit halves of the above
cudaError_t gemm_prepare_cg1(int bn, int smem_bytes);
cudaError_t gemm_launch_cg1(int bn, const KParams &p, int grid, int smem_bytes, cudaStream_t s);
cudaError_t gemm_prepare_cg2(int bn, int smem_bytes);
cudaError_t gemm_launch_cg2(int bn, const KParams &p, int grid, int smem_bytes, cudaStream_t s);
cudaError_t gemm_max_active_clusters_cg2(int bn, int smem_bytes, int *clusters);

// unfused comparison path: elementwise epilogue over an fp32 accumulator
cudaError_t ew_launch(const EwParams &p, int grid, cudaStream_t stream);
constexpr int kEwThreads = 256;

}  // namespace ge
