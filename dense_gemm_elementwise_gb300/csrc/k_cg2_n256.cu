// k_cg2_n256.cu -- fused kernel instances: cta_group::2, MMA N = 256.
#include "kernels_inst.cuh"

GE_INSTANTIATE_GEMM(2, 256, gemm_kernel_cg2_n256)
