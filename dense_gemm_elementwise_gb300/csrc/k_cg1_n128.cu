// k_cg1_n128.cu -- fused kernel instances: cta_group::1, MMA N = 128.
#include "kernels_inst.cuh"

GE_INSTANTIATE_GEMM(1, 128, gemm_kernel_cg1_n128)
