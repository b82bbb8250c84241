// k_cg1_n64.cu -- fused kernel instances: cta_group::1, MMA N = 64.
#include "kernels_inst.cuh"

GE_INSTANTIATE_GEMM(1, 64, gemm_kernel_cg1_n64)
