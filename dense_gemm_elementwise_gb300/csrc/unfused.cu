// unfused.cu -- the unfused comparison path ("Custom Epilogue Example",
// "Overview": a GEMM kernel followed by separate elementwise kernels, against
// one fused kernel that saves the memory traffic and the extra launches).
// Its second kernel: a grid-stride
// elementwise pass that reads the fp32 accumulator the GEMM wrote to a
// workspace, evaluates the same compiled epilogue program as the fused kernel
// (interpreter or catalog executor), and writes the outputs.  One thread
// handles 8 consecutive columns of one row (16-byte accesses); consecutive
// threads take consecutive column groups, so every warp access is contiguous.
// With M-major epilogue tensors consecutive threads take consecutive rows
// instead, so that each of a thread's 8 column accesses is contiguous across
// the warp.
#include <utility>

#include "catalog.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace ge {

struct GlobalMem {
  const EwParams *p;
  int64_t row;
  int col0;
  // element (row, col) of an M-major (L, N, M) tensor, row = l*M + i
  __device__ __forceinline__ int64_t col_index(int col) const {
    const int64_t l = row / p->M, i = row - l * p->M;
    return (l * p->N + col) * p->M + i;
  }
  template <int DT>
  __device__ __forceinline__ void aux(uint32_t i, float (&t)[kEwCols]) const {
    if (p->cd_m) {
#pragma unroll
      for (int e = 0; e < kEwCols; ++e)
        t[e] = col0 + e < p->N ? load_one<DT>(p->aux_ptr[i], col_index(col0 + e)) : 0.f;
      return;
    }
    const char *base = static_cast<const char *>(p->aux_ptr[i]) + row * p->N * (DT == GE_F32 ? 4 : 2);
    row_load<DT, kEwCols>(base, col0, p->N, t);
  }
  template <int DT>
  __device__ __forceinline__ void bcast(uint32_t i, float (&t)[kEwCols]) const {
    row_load<DT, kEwCols>(p->bcast_ptr[i], col0, p->N, t);
  }
  template <int DT>
  __device__ __forceinline__ void cbcast(uint32_t i, float (&t)[kEwCols]) const {
    const float v = load_one<DT>(p->cbcast_ptr[i], row % p->M);
#pragma unroll
    for (int e = 0; e < kEwCols; ++e) t[e] = v;
  }
  template <int DT>
  __device__ __forceinline__ void store(uint32_t o, const float (&t)[kEwCols]) const {
    if (p->cd_m) {
#pragma unroll
      for (int e = 0; e < kEwCols; ++e) {
        if (col0 + e >= p->N) break;
        const int64_t k = col_index(col0 + e);
        if constexpr (DT == GE_F32) static_cast<float *>(p->out_ptr[o])[k] = t[e];
        else if constexpr (DT == GE_BF16)
          static_cast<__nv_bfloat16 *>(p->out_ptr[o])[k] = __float2bfloat16_rn(t[e]);
        else static_cast<__half *>(p->out_ptr[o])[k] = __float2half_rn(t[e]);
      }
      return;
    }
    char *base = static_cast<char *>(p->out_ptr[o]) + row * p->N * (DT == GE_F32 ? 4 : 2);
    row_store<DT, kEwCols>(base, col0, p->N, t);
  }
};

template <class Epi>
__global__ void __launch_bounds__(kEwThreads) epilogue_elementwise_kernel(
    const __grid_constant__ EwParams p) {
  const int64_t units = p.rows * p.chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += stride) {
    int64_t row;
    int col0;
    if (p.cd_m) {
      const int64_t c = u / p.rows;
      row = u - c * p.rows;
      col0 = static_cast<int>(c) * kEwCols;
    } else {
      row = u / p.chunks_per_row;
      col0 = static_cast<int>(u - row * p.chunks_per_row) * kEwCols;
    }
    float acc[kEwCols];
    row_load<GE_F32, kEwCols>(p.acc + row * p.N, col0, p.N, acc);
    Epi::template run<kEwCols>(p.prog, acc, GlobalMem{&p, row, col0});
  }
}

template <size_t... K>
static const void *pick_ew(int epi, std::index_sequence<K...>) {
  static const void *const table[] = {reinterpret_cast<const void *>(
      &epilogue_elementwise_kernel<EpiStatic<catalog::Prog<K>>>)...};
  if (epi == -1) return reinterpret_cast<const void *>(&epilogue_elementwise_kernel<EpiInterpW<4, 4>>);
  if (epi == -2) return reinterpret_cast<const void *>(&epilogue_elementwise_kernel<EpiInterpW<4, 8>>);
  if (epi < 0) return nullptr;
  return epi < static_cast<int>(sizeof...(K)) ? table[epi] : nullptr;
}

const void *ew_kernel(int epi) { return pick_ew(epi, std::make_index_sequence<catalog::kCount>{}); }

}  // namespace ge
