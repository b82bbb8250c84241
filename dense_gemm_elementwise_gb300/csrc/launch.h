// launch.h -- kernel handles exported by the kernel translation units.
//
// Every handle is a __global__ function usable with cudaFuncSetAttribute and
// cudaLaunchKernelExC.  `epi` selects the epilogue executor: -1 the
// interpreter, k >= 0 the straight-line kernel of catalog entry k; `warps`
// the epilogue warps (4 or 8).  nullptr if not built.
#pragma once

#include <cuda_runtime_api.h>

#include <string>

#include "common.cuh"

namespace ge {

// fused GEMM + epilogue, (cta_group, BN) in {(1,64), (1,128), (1,256), (2,128), (2,256)}
const void *gemm_kernel_cg1_n64(int epi, int warps);
const void *gemm_kernel_cg1_n128(int epi, int warps);
const void *gemm_kernel_cg1_n256(int epi, int warps);
const void *gemm_kernel_cg2_n128(int epi, int warps);
const void *gemm_kernel_cg2_n256(int epi, int warps);

// a fused kernel compiled at run time for program P (nullptr, with the
// compiler's log in *log, if the runtime compiler is missing or fails)
const void *jit_gemm_kernel(const EpiProgram &P, int cg, int bn, int warps, std::string *log);
bool jit_available();

// unfused comparison path: elementwise epilogue over an fp32 accumulator
const void *ew_kernel(int epi);
constexpr int kEwThreads = 256;
constexpr int kEwCols = 8;  // columns per thread

}  // namespace ge
