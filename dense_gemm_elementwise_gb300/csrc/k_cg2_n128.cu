// k_cg2_n128.cu -- fused kernel instances: cta_group::2, MMA N = 128.
#include "kernels_inst.cuh"

GE_INSTANTIATE_GEMM(2, 128, gemm_kernel_cg2_n128)
