// unfused.cu -- the unfused comparison path's second kernel: a vectorised,
// grid-stride elementwise pass that reads the fp32 accumulator the GEMM wrote
// to a workspace, evaluates the same compiled epilogue program as the fused
// kernel, and writes the outputs.  One thread handles CH consecutive columns
// of one row; consecutive threads take consecutive column chunks.
#include "epilogue.cuh"
#include "launch.h"

namespace ge {

static __device__ __forceinline__ int esize(int dtype) { return dtype == GE_F32 ? 4 : 2; }

struct GlobalMem {
  const EwParams *p;
  int64_t row;
  int col0;
  __device__ __forceinline__ void aux(uint32_t i, float (&t)[CH]) const {
    const int dt = p->prog.tma_aux_dtype[i];
    const char *base = static_cast<const char *>(p->aux_ptr[i]) + row * p->N * esize(dt);
    row_load(base, dt, col0, p->N, t);
  }
  __device__ __forceinline__ void bcast(uint32_t i, float (&t)[CH]) const {
    row_load(p->bcast_ptr[i], p->prog.bcast_dtype[i], col0, p->N, t);
  }
  __device__ __forceinline__ void store(uint32_t o, const float (&t)[CH]) const {
    const int dt = p->prog.out_dtype[o];
    char *base = static_cast<char *>(p->out_ptr[o]) + row * p->N * esize(dt);
    row_store(base, dt, col0, p->N, t);
  }
};

__global__ void __launch_bounds__(kEwThreads) epilogue_elementwise_kernel(
    const __grid_constant__ EwParams p) {
  const int64_t units = p.rows * p.chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += stride) {
    const int64_t row = u / p.chunks_per_row;
    const int col0 = static_cast<int>(u - row * p.chunks_per_row) * CH;
    float acc[CH];
    row_load(p.acc + row * p.N, GE_F32, col0, p.N, acc);
    GlobalMem mem{&p, row, col0};
    run_program(p.prog, acc, mem);
  }
}

cudaError_t ew_launch(const EwParams &p, int grid, cudaStream_t stream) {
  epilogue_elementwise_kernel<<<grid, kEwThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ge
