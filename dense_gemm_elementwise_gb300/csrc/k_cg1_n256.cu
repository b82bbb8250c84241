// k_cg1_n256.cu -- fused kernel instances: cta_group::1, MMA N = 256.
#include "kernels_inst.cuh"

GE_INSTANTIATE_GEMM(1, 256, gemm_kernel_cg1_n256)
