// epilogue.cuh -- device interpreter of the compiled epilogue program.
//
// One call evaluates the whole program for one chunk: CH consecutive columns
// of one output row, held by one thread.  Instruction dispatch is uniform
// across the warp (every lane runs the same program), values stay in
// registers (all register-array indices are compile-time constants inside
// the switch cases), and every operation is plain fp32: multiply, add,
// max-with-zero.  A store rounds once, to nearest even, to its output type.
//
// The memory policy `Mem` supplies the leaves (aux tensors, broadcast
// vectors) and takes the stores: the fused kernel reads/writes swizzled
// shared-memory staging boxes moved by TMA; the unfused elementwise kernel
// reads/writes global memory directly.  The arithmetic is the same code in
// both, so the two paths agree bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"

namespace ge {

template <int N>
__device__ __forceinline__ void vcopy(float (&d)[N], const float (&s)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) d[i] = s[i];
}

// ------------------------------------------------------------ conversions --
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2 *>(&u);
  return __half22float2(h);
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t u) {
  // bf16 is the upper half of an fp32: widening is exact
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);  // cvt.rn: nearest even, a in the low half
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// 8 16-bit values in a uint4 -> 8 floats
__device__ __forceinline__ void unpack8(const uint4 &v, int dtype, float *t) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = (dtype == GE_BF16) ? bf16x2_to_f32x2(w[i]) : f16x2_to_f32x2(w[i]);
    t[2 * i] = f.x;
    t[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float *t, int dtype) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = (dtype == GE_BF16) ? f32x2_to_bf16x2(t[2 * i], t[2 * i + 1])
                              : f32x2_to_f16x2(t[2 * i], t[2 * i + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ----------------------------------------------------- swizzled staging box --
// A TMA box of 32 rows x CH columns.  Rows are 32 bytes (16-bit types, 32-byte
// swizzle) or 64 bytes (fp32, 64-byte swizzle); the swizzle XORs the 16-byte
// chunk index with address bits 7.. (row >> 2 or row >> 1), so a warp's 16-byte
// accesses to one chunk column touch every bank once per 8 threads.
__device__ __forceinline__ uint32_t box_off16(int row, int j) {
  return row * 32 + ((j ^ ((row >> 2) & 1)) << 4);
}
__device__ __forceinline__ uint32_t box_off32(int row, int j) {
  return row * 64 + ((j ^ ((row >> 1) & 3)) << 4);
}

__device__ __forceinline__ void box_load(const uint8_t *box, int dtype, int row, float (&t)[CH]) {
  if (dtype == GE_F32) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 v = *reinterpret_cast<const float4 *>(box + box_off32(row, j));
      t[4 * j] = v.x;
      t[4 * j + 1] = v.y;
      t[4 * j + 2] = v.z;
      t[4 * j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint4 v = *reinterpret_cast<const uint4 *>(box + box_off16(row, j));
      unpack8(v, dtype, t + 8 * j);
    }
  }
}

__device__ __forceinline__ void box_store(uint8_t *box, int dtype, int row, const float (&t)[CH]) {
  if (dtype == GE_F32) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4 *>(box + box_off32(row, j)) =
          make_float4(t[4 * j], t[4 * j + 1], t[4 * j + 2], t[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      *reinterpret_cast<uint4 *>(box + box_off16(row, j)) = pack8(t + 8 * j, dtype);
  }
}

// ------------------------------------------------------- global row access --
// CH elements of a row starting at column col0 (a multiple of CH).  Rows are
// multiples of 16 bytes and N is a multiple of 8, so each group of 8
// columns is entirely inside or entirely outside the row.
__device__ __forceinline__ void row_load(const void *row, int dtype, int col0, int N,
                                         float (&t)[CH]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = col0 + 8 * h;
    if (c < N) {
      if (dtype == GE_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(row) + c);
        float4 a = __ldg(p), b = __ldg(p + 1);
        t[8 * h] = a.x; t[8 * h + 1] = a.y; t[8 * h + 2] = a.z; t[8 * h + 3] = a.w;
        t[8 * h + 4] = b.x; t[8 * h + 5] = b.y; t[8 * h + 6] = b.z; t[8 * h + 7] = b.w;
      } else {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(row) + c));
        unpack8(v, dtype, t + 8 * h);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) t[8 * h + i] = 0.f;
    }
  }
}

__device__ __forceinline__ void row_store(void *row, int dtype, int col0, int N,
                                          const float (&t)[CH]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = col0 + 8 * h;
    if (c < N) {
      if (dtype == GE_F32) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(row) + c);
        p[0] = make_float4(t[8 * h], t[8 * h + 1], t[8 * h + 2], t[8 * h + 3]);
        p[1] = make_float4(t[8 * h + 4], t[8 * h + 5], t[8 * h + 6], t[8 * h + 7]);
      } else {
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(row) + c) = pack8(t + 8 * h, dtype);
      }
    }
  }
}

// ------------------------------------------------------------ interpreter --
template <class Mem>
__device__ __forceinline__ void run_program(const EpiProgram &P, const float (&acc)[CH], Mem &mem) {
  float r[kRegs][CH];
#pragma unroll
  for (int i = 0; i < kRegs; ++i)
#pragma unroll
    for (int e = 0; e < CH; ++e) r[i][e] = 0.f;

#pragma unroll 1
  for (int pc = 0; pc < P.n_ins; ++pc) {
    const uint32_t w = P.ins[pc];
    const uint32_t op = w & 0xFFu, dst = (w >> 8) & 0xFFu, src = (w >> 16) & 0xFFu, idx = w >> 24;
    float t[CH];
    switch (src) {
      case SRC_REG:
        switch (idx) {
          case 0: vcopy(t, r[0]); break;
          case 1: vcopy(t, r[1]); break;
          case 2: vcopy(t, r[2]); break;
          default: vcopy(t, r[3]); break;
        }
        break;
      case SRC_ACC: vcopy(t, acc); break;
      case SRC_AUX: mem.aux(idx, t); break;
      case SRC_BCAST: mem.bcast(idx, t); break;
      case SRC_SCALAR: {
        const float s = P.scalars[idx];
#pragma unroll
        for (int e = 0; e < CH; ++e) t[e] = s;
      } break;
      default:
#pragma unroll
        for (int e = 0; e < CH; ++e) t[e] = 0.f;
        break;
    }
#define GE_APPLY(D, EXPR)                     \
  case D: {                                   \
    _Pragma("unroll") for (int e = 0; e < CH; ++e) { \
      const float x = r[D][e];                \
      (void)x;                                \
      r[D][e] = (EXPR);                       \
    }                                         \
  } break;
    switch (op) {
      case OP_MOV:
        switch (dst) { GE_APPLY(0, t[e]) GE_APPLY(1, t[e]) GE_APPLY(2, t[e]) GE_APPLY(3, t[e]) }
        break;
      case OP_MUL:
        switch (dst) {
          GE_APPLY(0, __fmul_rn(x, t[e])) GE_APPLY(1, __fmul_rn(x, t[e]))
          GE_APPLY(2, __fmul_rn(x, t[e])) GE_APPLY(3, __fmul_rn(x, t[e]))
        }
        break;
      case OP_ADD:
        switch (dst) {
          GE_APPLY(0, __fadd_rn(x, t[e])) GE_APPLY(1, __fadd_rn(x, t[e]))
          GE_APPLY(2, __fadd_rn(x, t[e])) GE_APPLY(3, __fadd_rn(x, t[e]))
        }
        break;
      case OP_RELU:
        switch (dst) {
          GE_APPLY(0, x > 0.f ? x : 0.f) GE_APPLY(1, x > 0.f ? x : 0.f)
          GE_APPLY(2, x > 0.f ? x : 0.f) GE_APPLY(3, x > 0.f ? x : 0.f)
        }
        break;
      default:  // OP_STORE
        mem.store(dst, t);
        break;
    }
#undef GE_APPLY
  }
}

}  // namespace ge
