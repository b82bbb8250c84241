// k_cg2_n256_mc2.cu -- fused kernel instances: cta_group::2, MMA N = 256, two
// CTA pairs per cluster sharing A by TMA multicast.
#include "kernels_inst.cuh"

GE_INSTANTIATE_GEMM(2, 256, 2, gemm_kernel_cg2_n256_mc2)
