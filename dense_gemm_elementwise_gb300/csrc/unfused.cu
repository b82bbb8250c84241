// unfused.cu -- the unfused comparison path ("Custom Epilogue Example",
// "Overview": a GEMM kernel followed by separate elementwise kernels, against
// one fused kernel that saves the memory traffic and the extra launches).
// Its second kernel: a grid-stride
// elementwise pass that reads the fp32 accumulator the GEMM wrote to a
// workspace, evaluates the same compiled epilogue program as the fused kernel
// (interpreter or catalog executor), and writes the outputs.  One thread
// handles 8 consecutive elements along the contiguous dimension (16-byte
// accesses); consecutive threads take consecutive groups, so every warp
// access is contiguous.  The workspace is stored in the epilogue tensors'
// order: N-major (8 columns of one row per thread) or, with M-major epilogue
// tensors, M-major (8 rows of one column per thread).
#include <utility>

#include "catalog.cuh"
#include "epilogue.cuh"
#include "launch.h"

namespace ge {

// N-major tensors (L, M, N): 8 consecutive columns of one row per thread.
struct GlobalMem {
  const EwParams *p;
  int64_t row;
  int col0;
  template <int DT>
  __device__ __forceinline__ void aux(uint32_t i, float (&t)[kEwCols]) const {
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
    char *base = static_cast<char *>(p->out_ptr[o]) + row * p->N * (DT == GE_F32 ? 4 : 2);
    row_store<DT, kEwCols>(base, col0, p->N, t);
  }
};

// M-major tensors (L, N, M): 8 consecutive rows m0.. of one column per
// thread, the same 16-byte accesses along M.  An M-major plan has M*size a
// multiple of 16 bytes for some output, so M is a multiple of 4 and a group
// of 4 rows lies entirely inside or entirely outside the column.
template <int DT>
__device__ __forceinline__ void col_load8(const void *base, int64_t at, int m0, int M,
                                          float (&t)[kEwCols]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (m0 + 4 * h < M) {
      if constexpr (DT == GE_F32) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + at) + h);
        t[4 * h] = v.x; t[4 * h + 1] = v.y; t[4 * h + 2] = v.z; t[4 * h + 3] = v.w;
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + at) + h);
        const float2 a = DT == GE_BF16 ? bf16x2_to_f32x2(v.x) : f16x2_to_f32x2(v.x);
        const float2 b = DT == GE_BF16 ? bf16x2_to_f32x2(v.y) : f16x2_to_f32x2(v.y);
        t[4 * h] = a.x; t[4 * h + 1] = a.y; t[4 * h + 2] = b.x; t[4 * h + 3] = b.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) t[4 * h + i] = 0.f;
    }
  }
}

template <int DT>
__device__ __forceinline__ void col_store8(void *base, int64_t at, int m0, int M,
                                           const float (&t)[kEwCols]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (m0 + 4 * h < M) {
      if constexpr (DT == GE_F32) {
        reinterpret_cast<float4 *>(static_cast<float *>(base) + at)[h] =
            make_float4(t[4 * h], t[4 * h + 1], t[4 * h + 2], t[4 * h + 3]);
      } else {
        const uint32_t a = DT == GE_BF16 ? f32x2_to_bf16x2(t[4 * h], t[4 * h + 1])
                                         : f32x2_to_f16x2(t[4 * h], t[4 * h + 1]);
        const uint32_t b = DT == GE_BF16 ? f32x2_to_bf16x2(t[4 * h + 2], t[4 * h + 3])
                                         : f32x2_to_f16x2(t[4 * h + 2], t[4 * h + 3]);
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(base) + at)[h] = make_uint2(a, b);
      }
    }
  }
}

struct GlobalMemM {
  const EwParams *p;
  int64_t at;  // element index of (l, n, m0) in an (L, N, M) tensor
  int n, m0;
  template <int DT>
  __device__ __forceinline__ void aux(uint32_t i, float (&t)[kEwCols]) const {
    col_load8<DT>(p->aux_ptr[i], at, m0, p->M, t);
  }
  template <int DT>
  __device__ __forceinline__ void bcast(uint32_t i, float (&t)[kEwCols]) const {
    const float v = load_one<DT>(p->bcast_ptr[i], n);
#pragma unroll
    for (int e = 0; e < kEwCols; ++e) t[e] = v;
  }
  template <int DT>
  __device__ __forceinline__ void cbcast(uint32_t i, float (&t)[kEwCols]) const {
#pragma unroll
    for (int e = 0; e < kEwCols; ++e)
      t[e] = m0 + e < p->M ? load_one<DT>(p->cbcast_ptr[i], m0 + e) : 0.f;
  }
  template <int DT>
  __device__ __forceinline__ void store(uint32_t o, const float (&t)[kEwCols]) const {
    col_store8<DT>(p->out_ptr[o], at, m0, p->M, t);
  }
};

template <class Epi>
__global__ void __launch_bounds__(kEwThreads) epilogue_elementwise_kernel(
    const __grid_constant__ EwParams p) {
  const int64_t units = p.rows * p.chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += stride) {
    float acc[kEwCols];
    if (p.cd_m) {
      // units run along M within a column (l, n), columns after one another;
      // `rows` counts the L*N columns and `chunks_per_row` the 8-row groups
      const int64_t col = u / p.chunks_per_row;
      const int m0 = static_cast<int>(u - col * p.chunks_per_row) * kEwCols;
      const int64_t at = col * p.M + m0;
      col_load8<GE_F32>(p.acc, at, m0, p.M, acc);
      Epi::template run<kEwCols>(p.prog, acc,
                                 GlobalMemM{&p, at, static_cast<int>(col % p.N), m0});
    } else {
      const int64_t row = u / p.chunks_per_row;
      const int col0 = static_cast<int>(u - row * p.chunks_per_row) * kEwCols;
      row_load<GE_F32, kEwCols>(p.acc + row * p.N, col0, p.N, acc);
      Epi::template run<kEwCols>(p.prog, acc, GlobalMem{&p, row, col0});
    }
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
