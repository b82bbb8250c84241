// epilogue.cuh -- evaluation of the compiled epilogue program.
//
// Arithmetic as the pages fix it: every intermediate in fp32, one rounding
// per store ("Custom Epilogue Example", "Running the Example":
// --epi_dtype Float32); ReLU as where(d > 0, d, 0), so +0 for d <= 0
// ("Activation Functions"); the activations of the legacy interface's
// registry (the epilogue notebook of "CUTLASS Python 接口示例全解析"), with
// GELU in its exact erf form, written through erfc.
//
// A program (program.cuh) is evaluated for CH consecutive columns of one
// output row per thread.  Two executors evaluate the same instruction list:
//
//   run_program4<CH>         the interpreter: one uniform dispatch per
//   run_programR<CH, R>      instruction per CH columns (any DAG the plan
//                            compiler accepts; programs needing more than 4
//                            registers use the R = kRegs variant);
//   run_static_from<SP,..>   the catalog executor: the instruction list is a
//                            compile-time constant, every dispatch is resolved
//                            by `if constexpr`, leaving straight-line fp32 code.
//
// All register-array indices are compile-time constants (a run-time register
// number selects among them through a switch), so values stay in registers.  Multiplies and adds are __fmul_rn/__fadd_rn (never contracted
// into an FMA); ReLU returns +0 for x <= 0; a store rounds once to nearest
// even.  The memory policy `Mem` supplies aux tensors and broadcast vectors
// and takes the stores: swizzled shared-memory TMA boxes in the fused kernel,
// global memory in the unfused elementwise kernel.  Same arithmetic, same
// order, so every executor and kernel agrees bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

template <int DT>
__device__ __forceinline__ void unpack8(const uint4 &v, float *t) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = DT == GE_BF16 ? bf16x2_to_f32x2(w[i]) : f16x2_to_f32x2(w[i]);
    t[2 * i] = f.x;
    t[2 * i + 1] = f.y;
  }
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float *t) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = DT == GE_BF16 ? f32x2_to_bf16x2(t[2 * i], t[2 * i + 1])
                         : f32x2_to_f16x2(t[2 * i], t[2 * i + 1]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ----------------------------------------------------- swizzled staging box --
// One TMA box: kEpiRows (128) rows x EW (32) columns; a warp touches the 32
// rows of its lane quarter (row = 32 * quarter + lane).  16-bit rows are 64 bytes
// (64-byte swizzle: 16-byte chunk j of row r at r*64 + ((j ^ ((r>>1)&3))*16));
// fp32 rows are 128 bytes (128-byte swizzle: chunk j at r*128 + ((j ^ (r&7))*16)).
// Either way the 8 lanes of a 16-byte access phase hit 8 different bank
// groups.  `half` selects columns [16*half, 16*half + 16) of the box.
template <int DT>
__device__ __forceinline__ void box_load(const uint8_t *box, int row, int half, float (&t)[16]) {
  if constexpr (DT == GE_F32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * half + k;
      const float4 v = *reinterpret_cast<const float4 *>(box + row * 128 + ((j ^ (row & 7)) << 4));
      t[4 * k] = v.x;
      t[4 * k + 1] = v.y;
      t[4 * k + 2] = v.z;
      t[4 * k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = 2 * half + k;
      const uint4 v =
          *reinterpret_cast<const uint4 *>(box + row * 64 + ((j ^ ((row >> 1) & 3)) << 4));
      unpack8<DT>(v, t + 8 * k);
    }
  }
}

template <int DT>
__device__ __forceinline__ void box_store(uint8_t *box, int row, int half, const float (&t)[16]) {
  if constexpr (DT == GE_F32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = 4 * half + k;
      *reinterpret_cast<float4 *>(box + row * 128 + ((j ^ (row & 7)) << 4)) =
          make_float4(t[4 * k], t[4 * k + 1], t[4 * k + 2], t[4 * k + 3]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = 2 * half + k;
      *reinterpret_cast<uint4 *>(box + row * 64 + ((j ^ ((row >> 1) & 3)) << 4)) =
          pack8<DT>(t + 8 * k);
    }
  }
}

// Epilogue tensors stored M-major (each batch column-major): the staged box
// is 32 columns of kEpiRows rows, a column's rows contiguous ([n][m], no
// swizzle).  Lane = row touches one element per column, so every warp access
// covers a contiguous 64- or 128-byte run of a column without bank conflicts.
__device__ __forceinline__ float widen16(uint16_t u, bool bf16) {
  return bf16 ? __uint_as_float(static_cast<uint32_t>(u) << 16)
              : __half2float(__ushort_as_half(static_cast<unsigned short>(u)));
}

template <int DT>
__device__ __forceinline__ void col_box_load(const uint8_t *box, int row, int half, float (&t)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int n = 16 * half + e;
    if constexpr (DT == GE_F32)
      t[e] = reinterpret_cast<const float *>(box)[n * kEpiRows + row];
    else
      t[e] = widen16(reinterpret_cast<const uint16_t *>(box)[n * kEpiRows + row], DT == GE_BF16);
  }
}

template <int DT>
__device__ __forceinline__ void col_box_store(uint8_t *box, int row, int half, const float (&t)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int n = 16 * half + e;
    if constexpr (DT == GE_F32) {
      reinterpret_cast<float *>(box)[n * kEpiRows + row] = t[e];
    } else if constexpr (DT == GE_BF16) {
      reinterpret_cast<__nv_bfloat16 *>(box)[n * kEpiRows + row] = __float2bfloat16_rn(t[e]);
    } else {
      reinterpret_cast<__half *>(box)[n * kEpiRows + row] = __float2half_rn(t[e]);
    }
  }
}

// ------------------------------------------------------- global row access --
// C (8 or 16) elements of a row starting at column col0 (a multiple of 8).
// Rows are multiples of 16 bytes and N is a multiple of 8, so each group of 8
// columns is entirely inside or entirely outside the row.
template <int DT, int C>
__device__ __forceinline__ void row_load(const void *row, int col0, int N, float (&t)[C]) {
#pragma unroll
  for (int h = 0; h < C / 8; ++h) {
    const int c = col0 + 8 * h;
    if (c < N) {
      if constexpr (DT == GE_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(row) + c);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        t[8 * h] = a.x; t[8 * h + 1] = a.y; t[8 * h + 2] = a.z; t[8 * h + 3] = a.w;
        t[8 * h + 4] = b.x; t[8 * h + 5] = b.y; t[8 * h + 6] = b.z; t[8 * h + 7] = b.w;
      } else {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(row) + c));
        unpack8<DT>(v, t + 8 * h);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) t[8 * h + i] = 0.f;
    }
  }
}

template <int DT, int C>
__device__ __forceinline__ void row_store(void *row, int col0, int N, const float (&t)[C]) {
#pragma unroll
  for (int h = 0; h < C / 8; ++h) {
    const int c = col0 + 8 * h;
    if (c < N) {
      if constexpr (DT == GE_F32) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(row) + c);
        p[0] = make_float4(t[8 * h], t[8 * h + 1], t[8 * h + 2], t[8 * h + 3]);
        p[1] = make_float4(t[8 * h + 4], t[8 * h + 5], t[8 * h + 6], t[8 * h + 7]);
      } else {
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(row) + c) = pack8<DT>(t + 8 * h);
      }
    }
  }
}

// one element of a vector, widened to fp32 (column-broadcast values)
template <int DT>
__device__ __forceinline__ float load_one(const void *base, int64_t i) {
  if constexpr (DT == GE_F32) {
    return __ldg(static_cast<const float *>(base) + i);
  } else {
    const uint32_t u = __ldg(static_cast<const uint16_t *>(base) + i);
    return DT == GE_BF16 ? __uint_as_float(u << 16) : __half2float(__ushort_as_half(static_cast<unsigned short>(u)));
  }
}

// run-time element type -> compile-time instantiation
#define GE_DISPATCH_DTYPE(dt, CALL) \
  do {                              \
    if ((dt) == GE_F32) {           \
      constexpr int DT_ = GE_F32;   \
      CALL;                         \
    } else if ((dt) == GE_BF16) {   \
      constexpr int DT_ = GE_BF16;  \
      CALL;                         \
    } else {                        \
      constexpr int DT_ = GE_F16;   \
      CALL;                         \
    }                               \
  } while (0)

// ------------------------------------------------------------ activations --
// fp32 evaluations of the activation registry's functions through the CUDA
// math library (expf, tanhf, erfcf); every other step correctly rounded.
constexpr float kRsqrt2 = 0.70710678118654752440f;  // 1/sqrt(2)

__device__ __forceinline__ float act_sigmoid(float x) { return __fdiv_rn(1.f, __fadd_rn(1.f, expf(-x))); }
__device__ __forceinline__ float act_tanh(float x) { return tanhf(x); }
// 1 + erf(z) = erfc(-z); erfc keeps the relative accuracy of the far
// negative tail, where 1 + erf(z) cancels to 0
__device__ __forceinline__ float act_gelu(float x) {
  return __fmul_rn(__fmul_rn(0.5f, x), erfcf(__fmul_rn(-x, kRsqrt2)));
}
__device__ __forceinline__ float act_silu(float x) { return __fdiv_rn(x, __fadd_rn(1.f, expf(-x))); }
__device__ __forceinline__ float act_hardswish(float x) {
  const float c = fminf(fmaxf(__fadd_rn(x, 3.f), 0.f), 6.f);
  return __fdiv_rn(__fmul_rn(x, c), 6.f);
}

template <uint32_t OP>
__device__ __forceinline__ float activation(float x) {
  if constexpr (OP == OP_SIGMOID) return act_sigmoid(x);
  else if constexpr (OP == OP_TANH) return act_tanh(x);
  else if constexpr (OP == OP_GELU) return act_gelu(x);
  else if constexpr (OP == OP_SILU) return act_silu(x);
  else return act_hardswish(x);
}

template <uint32_t OP, int C>
__device__ __forceinline__ void activation_vec(float (&t)[C]) {
#pragma unroll
  for (int e = 0; e < C; ++e) t[e] = activation<OP>(t[e]);
}

__host__ __device__ constexpr bool is_activation_op(uint32_t op) {
  return op == OP_SIGMOID || op == OP_TANH || op == OP_GELU || op == OP_SILU || op == OP_HARDSWISH;
}

// ------------------------------------------------------------ interpreter --
// Four program registers: every operation has its own switch over the
// destination register (fewest live values, no spills at 4 warps).
template <int C, class Mem>
__device__ __forceinline__ void run_program4(const EpiProgram &P, const float (&acc)[C], const Mem &mem) {
  float r[4][C];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < C; ++e) r[i][e] = 0.f;

#pragma unroll 1
  for (int pc = 0; pc < P.n_ins; ++pc) {
    const uint32_t w = P.ins[pc];
    const uint32_t op = w & 0xFFu, dst = (w >> 8) & 0xFFu, src = (w >> 16) & 0xFFu, idx = w >> 24;
    float t[C];
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
      case SRC_AUX: GE_DISPATCH_DTYPE(P.tma_aux_dtype[idx], mem.template aux<DT_>(idx, t)); break;
      case SRC_BCAST: GE_DISPATCH_DTYPE(P.bcast_dtype[idx], mem.template bcast<DT_>(idx, t)); break;
      case SRC_CBCAST: GE_DISPATCH_DTYPE(P.cbcast_dtype[idx], mem.template cbcast<DT_>(idx, t)); break;
      case SRC_SCALAR: {
        const float s = P.scalars[idx];
#pragma unroll
        for (int e = 0; e < C; ++e) t[e] = s;
      } break;
      default:
#pragma unroll
        for (int e = 0; e < C; ++e) t[e] = 0.f;
        break;
    }
#define GE_APPLY(D, EXPR)                             \
  case D: {                                           \
    _Pragma("unroll") for (int e = 0; e < C; ++e) {   \
      const float x = r[D][e];                        \
      (void)x;                                        \
      r[D][e] = (EXPR);                               \
    }                                                 \
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
      case OP_SUB:
        switch (dst) {
          GE_APPLY(0, __fsub_rn(x, t[e])) GE_APPLY(1, __fsub_rn(x, t[e]))
          GE_APPLY(2, __fsub_rn(x, t[e])) GE_APPLY(3, __fsub_rn(x, t[e]))
        }
        break;
      case OP_RSUB:
        switch (dst) {
          GE_APPLY(0, __fsub_rn(t[e], x)) GE_APPLY(1, __fsub_rn(t[e], x))
          GE_APPLY(2, __fsub_rn(t[e], x)) GE_APPLY(3, __fsub_rn(t[e], x))
        }
        break;
      case OP_DIV:
        switch (dst) {
          GE_APPLY(0, __fdiv_rn(x, t[e])) GE_APPLY(1, __fdiv_rn(x, t[e]))
          GE_APPLY(2, __fdiv_rn(x, t[e])) GE_APPLY(3, __fdiv_rn(x, t[e]))
        }
        break;
      case OP_RDIV:
        switch (dst) {
          GE_APPLY(0, __fdiv_rn(t[e], x)) GE_APPLY(1, __fdiv_rn(t[e], x))
          GE_APPLY(2, __fdiv_rn(t[e], x)) GE_APPLY(3, __fdiv_rn(t[e], x))
        }
        break;
      case OP_MIN:
        switch (dst) {
          GE_APPLY(0, fminf(x, t[e])) GE_APPLY(1, fminf(x, t[e]))
          GE_APPLY(2, fminf(x, t[e])) GE_APPLY(3, fminf(x, t[e]))
        }
        break;
      case OP_MAX:
        switch (dst) {
          GE_APPLY(0, fmaxf(x, t[e])) GE_APPLY(1, fmaxf(x, t[e]))
          GE_APPLY(2, fmaxf(x, t[e])) GE_APPLY(3, fmaxf(x, t[e]))
        }
        break;
      case OP_LEAKY:
        switch (dst) {
          GE_APPLY(0, x > 0.f ? x : __fmul_rn(t[e], x)) GE_APPLY(1, x > 0.f ? x : __fmul_rn(t[e], x))
          GE_APPLY(2, x > 0.f ? x : __fmul_rn(t[e], x)) GE_APPLY(3, x > 0.f ? x : __fmul_rn(t[e], x))
        }
        break;
      case OP_RLEAKY:
        switch (dst) {
          GE_APPLY(0, t[e] > 0.f ? t[e] : __fmul_rn(x, t[e]))
          GE_APPLY(1, t[e] > 0.f ? t[e] : __fmul_rn(x, t[e]))
          GE_APPLY(2, t[e] > 0.f ? t[e] : __fmul_rn(x, t[e]))
          GE_APPLY(3, t[e] > 0.f ? t[e] : __fmul_rn(x, t[e]))
        }
        break;
      case OP_SIGMOID:
      case OP_TANH:
      case OP_GELU:
      case OP_SILU:
      case OP_HARDSWISH:
        // one copy of each activation's code, applied to the fetched operand
        switch (op) {
          case OP_SIGMOID: activation_vec<OP_SIGMOID>(t); break;
          case OP_TANH: activation_vec<OP_TANH>(t); break;
          case OP_GELU: activation_vec<OP_GELU>(t); break;
          case OP_SILU: activation_vec<OP_SILU>(t); break;
          default: activation_vec<OP_HARDSWISH>(t); break;
        }
        switch (dst) { GE_APPLY(0, t[e]) GE_APPLY(1, t[e]) GE_APPLY(2, t[e]) GE_APPLY(3, t[e]) }
        break;
      default:  // OP_STORE
        GE_DISPATCH_DTYPE(P.out_dtype[dst], mem.template store<DT_>(dst, t));
        break;
    }
#undef GE_APPLY
  }
}

// More program registers (up to kRegs): a register is selected at run time: a register is read into, or
// written from, a plain vector through one switch, so each operation's code
// exists once, whatever register it works on.
#define GE_REG_CASE(I, STMT) \
  case I:                    \
    if constexpr (I < R) {   \
      STMT;                  \
    }                        \
    break;

template <int R, int C>
__device__ __forceinline__ void reg_read(const float (&r)[R][C], uint32_t k, float (&t)[C]) {
  switch (k) {
    GE_REG_CASE(0, vcopy(t, r[0])) GE_REG_CASE(1, vcopy(t, r[1])) GE_REG_CASE(2, vcopy(t, r[2]))
    GE_REG_CASE(3, vcopy(t, r[3])) GE_REG_CASE(4, vcopy(t, r[4])) GE_REG_CASE(5, vcopy(t, r[5]))
    GE_REG_CASE(6, vcopy(t, r[6])) GE_REG_CASE(7, vcopy(t, r[7]))
    default: break;
  }
}

template <int R, int C>
__device__ __forceinline__ void reg_write(float (&r)[R][C], uint32_t k, const float (&t)[C]) {
  switch (k) {
    GE_REG_CASE(0, vcopy(r[0], t)) GE_REG_CASE(1, vcopy(r[1], t)) GE_REG_CASE(2, vcopy(r[2], t))
    GE_REG_CASE(3, vcopy(r[3], t)) GE_REG_CASE(4, vcopy(r[4], t)) GE_REG_CASE(5, vcopy(r[5], t))
    GE_REG_CASE(6, vcopy(r[6], t)) GE_REG_CASE(7, vcopy(r[7], t))
    default: break;
  }
}
#undef GE_REG_CASE

// R: program registers the kernel holds (kRegs for programs that need more
// than 4)
template <int C, int R, class Mem>
__device__ __forceinline__ void run_programR(const EpiProgram &P, const float (&acc)[C], const Mem &mem) {
  static_assert(R <= kRegs, "program registers");
  float r[R][C];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int e = 0; e < C; ++e) r[i][e] = 0.f;

#pragma unroll 1
  for (int pc = 0; pc < P.n_ins; ++pc) {
    const uint32_t w = P.ins[pc];
    const uint32_t op = w & 0xFFu, dst = (w >> 8) & 0xFFu, src = (w >> 16) & 0xFFu, idx = w >> 24;
    float t[C];
    switch (src) {
      case SRC_REG: reg_read(r, idx, t); break;
      case SRC_ACC: vcopy(t, acc); break;
      case SRC_AUX: GE_DISPATCH_DTYPE(P.tma_aux_dtype[idx], mem.template aux<DT_>(idx, t)); break;
      case SRC_BCAST: GE_DISPATCH_DTYPE(P.bcast_dtype[idx], mem.template bcast<DT_>(idx, t)); break;
      case SRC_CBCAST: GE_DISPATCH_DTYPE(P.cbcast_dtype[idx], mem.template cbcast<DT_>(idx, t)); break;
      case SRC_SCALAR: {
        const float s = P.scalars[idx];
#pragma unroll
        for (int e = 0; e < C; ++e) t[e] = s;
      } break;
      default:
#pragma unroll
        for (int e = 0; e < C; ++e) t[e] = 0.f;
        break;
    }
    if (op == OP_STORE) {
      GE_DISPATCH_DTYPE(P.out_dtype[dst], mem.template store<DT_>(dst, t));
      continue;
    }
    // u: the destination register's value, updated in place
    float u[C];
    if (op != OP_MOV && !is_activation_op(op)) reg_read(r, dst, u);
#define GE_EACH(EXPR)                                      \
  {                                                        \
    _Pragma("unroll") for (int e = 0; e < C; ++e) {        \
      const float x = u[e];                                \
      (void)x;                                             \
      u[e] = (EXPR);                                       \
    }                                                      \
  }
    switch (op) {
      case OP_MOV: vcopy(u, t); break;
      case OP_MUL: GE_EACH(__fmul_rn(x, t[e])) break;
      case OP_ADD: GE_EACH(__fadd_rn(x, t[e])) break;
      case OP_RELU: GE_EACH(x > 0.f ? x : 0.f) break;
      case OP_SUB: GE_EACH(__fsub_rn(x, t[e])) break;
      case OP_RSUB: GE_EACH(__fsub_rn(t[e], x)) break;
      case OP_DIV: GE_EACH(__fdiv_rn(x, t[e])) break;
      case OP_RDIV: GE_EACH(__fdiv_rn(t[e], x)) break;
      case OP_MIN: GE_EACH(fminf(x, t[e])) break;
      case OP_MAX: GE_EACH(fmaxf(x, t[e])) break;
      case OP_LEAKY: GE_EACH(x > 0.f ? x : __fmul_rn(t[e], x)) break;
      case OP_RLEAKY: GE_EACH(t[e] > 0.f ? t[e] : __fmul_rn(x, t[e])) break;
      case OP_SIGMOID: vcopy(u, t); activation_vec<OP_SIGMOID>(u); break;
      case OP_TANH: vcopy(u, t); activation_vec<OP_TANH>(u); break;
      case OP_GELU: vcopy(u, t); activation_vec<OP_GELU>(u); break;
      case OP_SILU: vcopy(u, t); activation_vec<OP_SILU>(u); break;
      default: vcopy(u, t); activation_vec<OP_HARDSWISH>(u); break;
    }
#undef GE_EACH
    reg_write(r, dst, u);
  }
}

// ---------------------------------------------------- catalog (static) --
template <class SP, int PC, int C, class Mem>
__device__ __forceinline__ void run_static_from(float (&r)[kRegs][C], const float (&acc)[C],
                                                const Mem &mem, const float *scalars) {
  if constexpr (PC < SP::P.n_ins) {
    constexpr uint32_t w = SP::P.ins[PC];
    constexpr uint32_t op = w & 0xFFu, dst = (w >> 8) & 0xFFu, src = (w >> 16) & 0xFFu,
                       idx = w >> 24;
    if constexpr (op == OP_RELU) {
#pragma unroll
      for (int e = 0; e < C; ++e) r[dst][e] = r[dst][e] > 0.f ? r[dst][e] : 0.f;
    } else {
      float t[C];
      if constexpr (src == SRC_REG) {
        vcopy(t, r[idx]);
      } else if constexpr (src == SRC_ACC) {
        vcopy(t, acc);
      } else if constexpr (src == SRC_AUX) {
        mem.template aux<SP::P.tma_aux_dtype[idx]>(idx, t);
      } else if constexpr (src == SRC_BCAST) {
        mem.template bcast<SP::P.bcast_dtype[idx]>(idx, t);
      } else if constexpr (src == SRC_CBCAST) {
        mem.template cbcast<SP::P.cbcast_dtype[idx]>(idx, t);
      } else {
        const float s = scalars[idx];
#pragma unroll
        for (int e = 0; e < C; ++e) t[e] = s;
      }
      if constexpr (op == OP_MOV) {
        vcopy(r[dst], t);
      } else if constexpr (op == OP_MUL) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = __fmul_rn(r[dst][e], t[e]);
      } else if constexpr (op == OP_ADD) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = __fadd_rn(r[dst][e], t[e]);
      } else if constexpr (op == OP_SUB) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = __fsub_rn(r[dst][e], t[e]);
      } else if constexpr (op == OP_RSUB) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = __fsub_rn(t[e], r[dst][e]);
      } else if constexpr (op == OP_DIV) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = __fdiv_rn(r[dst][e], t[e]);
      } else if constexpr (op == OP_RDIV) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = __fdiv_rn(t[e], r[dst][e]);
      } else if constexpr (op == OP_MIN) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = fminf(r[dst][e], t[e]);
      } else if constexpr (op == OP_MAX) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = fmaxf(r[dst][e], t[e]);
      } else if constexpr (op == OP_LEAKY) {
#pragma unroll
        for (int e = 0; e < C; ++e)
          r[dst][e] = r[dst][e] > 0.f ? r[dst][e] : __fmul_rn(t[e], r[dst][e]);
      } else if constexpr (op == OP_RLEAKY) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = t[e] > 0.f ? t[e] : __fmul_rn(r[dst][e], t[e]);
      } else if constexpr (is_activation_op(op)) {
#pragma unroll
        for (int e = 0; e < C; ++e) r[dst][e] = activation<op>(t[e]);
      } else {
        mem.template store<SP::P.out_dtype[dst]>(dst, t);
      }
    }
    run_static_from<SP, PC + 1, C>(r, acc, mem, scalars);
  }
}

// Epilogue selectors used as kernel template arguments.
// kWarps: epilogue warps of the fused kernels built with the selector (the
// unfused elementwise kernel ignores it).
template <int W = 4, int R = 4>
struct EpiInterpW {
  static constexpr int kWarps = W;
  template <int C, class Mem>
  __device__ __forceinline__ static void run(const EpiProgram &P, const float (&acc)[C], const Mem &mem) {
    if constexpr (R == 4) run_program4<C>(P, acc, mem);
    else run_programR<C, R>(P, acc, mem);
  }
};
using EpiInterp = EpiInterpW<4>;

template <class SP, int W = 4>
struct EpiStatic {
  static constexpr int kWarps = W;
  template <int C, class Mem>
  __device__ __forceinline__ static void run(const EpiProgram &P, const float (&acc)[C], const Mem &mem) {
    float r[kRegs][C] = {};
    run_static_from<SP, 0, C>(r, acc, mem, P.scalars);
  }
};

}  // namespace ge
