// program.cuh -- the DAG -> epilogue-program compiler.
//
// The DAG is the one "CUTLASS Operator API: Custom epilogue fusions for
// GEMMs" describes ("How the epilogue fusion API works", figure
// "Intermediate DAG representation"): AccFetch, Load and compute nodes
// ending in Stores, in single-assignment order ("Defining an epilogue via a
// Python function").
//
// constexpr and __host__ __device__ so that the very same function compiles
// user DAGs at plan time (host) and the built-in catalog of epilogues at
// build time (template arguments of the specialised kernels).  A user DAG
// whose compiled program equals a catalog entry runs the straight-line
// kernel for that entry; any other DAG runs the interpreter kernel.  Both
// evaluate the identical instruction list in the identical order, so they
// agree bit for bit.
#pragma once

#include "common.cuh"

namespace ge {

// Ranking of leaf sources for commutative operand order: a two-operand op
// that needs a fresh register moves the lower-ranked operand in first, so
// mul(alpha, accum) and mul(accum, alpha) compile to the same program
// (fp32 multiply and add are commutative bit for bit).
__host__ __device__ constexpr int src_rank(uint32_t src) {
  return src == SRC_ACC      ? 0
         : src == SRC_AUX    ? 1
         : src == SRC_BCAST  ? 2
         : src == SRC_CBCAST ? 3
         : src == SRC_REG    ? 4
                             : 5;
}

__host__ __device__ constexpr bool is_binary(int op) {
  return op == GE_MUL || op == GE_ADD || op == GE_SUB || op == GE_DIV || op == GE_MIN ||
         op == GE_MAX || op == GE_LEAKY_RELU;
}

// activations compiled as r[dst] = f(src)
__host__ __device__ constexpr bool is_activation(int op) {
  return op == GE_SIGMOID || op == GE_TANH || op == GE_GELU || op == GE_SILU ||
         op == GE_HARDSWISH;
}

struct CompileResult {
  int status;
  EpiProgram prog;
};

// Greedy register allocation in node order.  Leaves are never copied into a
// register unless an operation needs a destination for them; an operation
// reuses an operand's register in place when this is the operand's last use.
// Assumes a DAG that passed validation.
__host__ __device__ constexpr CompileResult compile_program(const ge_dtypes &dt, const ge_dag &dag) {
  CompileResult R{GE_OK, EpiProgram{}};
  EpiProgram &P = R.prog;
  const int n = dag.n;
  int last_use[GE_MAX_NODES] = {};
  for (int i = 0; i < GE_MAX_NODES; ++i) last_use[i] = -1;
  for (int i = 0; i < n; ++i) {
    const ge_node &nd = dag.node[i];
    if (is_binary(nd.op)) {
      last_use[nd.a] = i;
      last_use[nd.b] = i;
    } else if (nd.op == GE_RELU || nd.op == GE_STORE || is_activation(nd.op)) {
      last_use[nd.a] = i;
    }
  }
  int tma_of_slot[GE_MAX_AUX] = {};
  int bc_of_slot[GE_MAX_AUX] = {};
  int cb_of_slot[GE_MAX_AUX] = {};
  for (int s = 0; s < GE_MAX_AUX; ++s) tma_of_slot[s] = bc_of_slot[s] = cb_of_slot[s] = -1;
  uint32_t loc_src[GE_MAX_NODES] = {};
  uint32_t loc_idx[GE_MAX_NODES] = {};
  bool busy[kRegs] = {};
  int max_regs = 0;

  for (int i = 0; i < n; ++i) {
    const ge_node &nd = dag.node[i];
    if (P.n_ins + 2 > kMaxIns) {
      R.status = GE_ERR_UNSUPPORTED;
      return R;
    }
    switch (nd.op) {
      case GE_ACCFETCH:
        loc_src[i] = SRC_ACC;
        loc_idx[i] = 0;
        break;
      case GE_LOAD: {
        if (tma_of_slot[nd.slot] < 0) {
          if (P.n_tma_aux >= GE_MAX_TMA_AUX) {
            R.status = GE_ERR_UNSUPPORTED;
            return R;
          }
          tma_of_slot[nd.slot] = P.n_tma_aux;
          P.tma_aux_slot[P.n_tma_aux] = nd.slot;
          P.tma_aux_dtype[P.n_tma_aux] = dt.aux[nd.slot];
          ++P.n_tma_aux;
        }
        loc_src[i] = SRC_AUX;
        loc_idx[i] = static_cast<uint32_t>(tma_of_slot[nd.slot]);
        break;
      }
      case GE_BROADCAST: {
        if (bc_of_slot[nd.slot] < 0) {
          bc_of_slot[nd.slot] = P.n_bcast;
          P.bcast_slot[P.n_bcast] = nd.slot;
          P.bcast_dtype[P.n_bcast] = dt.aux[nd.slot];
          ++P.n_bcast;
        }
        loc_src[i] = SRC_BCAST;
        loc_idx[i] = static_cast<uint32_t>(bc_of_slot[nd.slot]);
        break;
      }
      case GE_COL_BROADCAST: {
        if (cb_of_slot[nd.slot] < 0) {
          cb_of_slot[nd.slot] = P.n_cbcast;
          P.cbcast_slot[P.n_cbcast] = nd.slot;
          P.cbcast_dtype[P.n_cbcast] = dt.aux[nd.slot];
          ++P.n_cbcast;
        }
        loc_src[i] = SRC_CBCAST;
        loc_idx[i] = static_cast<uint32_t>(cb_of_slot[nd.slot]);
        break;
      }
      case GE_SCALAR:
        loc_src[i] = SRC_SCALAR;
        loc_idx[i] = static_cast<uint32_t>(nd.slot);
        break;
      case GE_MUL:
      case GE_ADD:
      case GE_SUB:
      case GE_DIV:
      case GE_MIN:
      case GE_MAX:
      case GE_LEAKY_RELU: {
        // two-address forms; subtraction, division and leaky ReLU have a
        // reversed form for when the second operand's register is the one
        // reused
        const bool commutes = nd.op == GE_MUL || nd.op == GE_ADD || nd.op == GE_MIN ||
                              nd.op == GE_MAX;
        const uint32_t op = nd.op == GE_MUL   ? OP_MUL
                            : nd.op == GE_ADD ? OP_ADD
                            : nd.op == GE_SUB ? OP_SUB
                            : nd.op == GE_DIV ? OP_DIV
                            : nd.op == GE_MIN ? OP_MIN
                            : nd.op == GE_MAX ? OP_MAX
                                              : OP_LEAKY;
        const uint32_t rop = nd.op == GE_SUB          ? OP_RSUB
                             : nd.op == GE_DIV        ? OP_RDIV
                             : nd.op == GE_LEAKY_RELU ? OP_RLEAKY
                                                      : op;
        const bool a_dies = loc_src[nd.a] == SRC_REG && last_use[nd.a] == i;
        const bool b_dies = loc_src[nd.b] == SRC_REG && last_use[nd.b] == i;
        int d = -1, other = -1;
        uint32_t emit_op = op;
        if (a_dies && (!b_dies || loc_idx[nd.a] <= loc_idx[nd.b] || !commutes)) {
          d = static_cast<int>(loc_idx[nd.a]);
          other = nd.b;
        } else if (b_dies) {
          d = static_cast<int>(loc_idx[nd.b]);
          other = nd.a;
          emit_op = rop;
        } else {
          for (int r = 0; r < kRegs; ++r)
            if (!busy[r]) {
              d = r;
              break;
            }
          if (d < 0) {
            R.status = GE_ERR_UNSUPPORTED;
            return R;
          }
          busy[d] = true;
          if (d + 1 > max_regs) max_regs = d + 1;
          int first = nd.a;
          other = nd.b;
          const int ra = src_rank(loc_src[nd.a]), rb = src_rank(loc_src[nd.b]);
          if (commutes && (rb < ra || (rb == ra && loc_idx[nd.b] < loc_idx[nd.a]))) {
            first = nd.b;
            other = nd.a;
          }
          P.ins[P.n_ins++] = pack_ins(OP_MOV, static_cast<uint32_t>(d), loc_src[first], loc_idx[first]);
        }
        P.ins[P.n_ins++] =
            pack_ins(emit_op, static_cast<uint32_t>(d), loc_src[other], loc_idx[other]);
        const int refs[2] = {nd.a, nd.b};
        for (int k = 0; k < 2; ++k) {
          const int ref = refs[k];
          if (loc_src[ref] == SRC_REG && last_use[ref] == i && static_cast<int>(loc_idx[ref]) != d)
            busy[loc_idx[ref]] = false;
        }
        loc_src[i] = SRC_REG;
        loc_idx[i] = static_cast<uint32_t>(d);
        if (last_use[i] < 0) busy[d] = false;  // dead value
        break;
      }
      case GE_RELU: {
        int d = -1;
        if (loc_src[nd.a] == SRC_REG && last_use[nd.a] == i) {
          d = static_cast<int>(loc_idx[nd.a]);
        } else {
          for (int r = 0; r < kRegs; ++r)
            if (!busy[r]) {
              d = r;
              break;
            }
          if (d < 0) {
            R.status = GE_ERR_UNSUPPORTED;
            return R;
          }
          busy[d] = true;
          if (d + 1 > max_regs) max_regs = d + 1;
          P.ins[P.n_ins++] = pack_ins(OP_MOV, static_cast<uint32_t>(d), loc_src[nd.a], loc_idx[nd.a]);
        }
        P.ins[P.n_ins++] = pack_ins(OP_RELU, static_cast<uint32_t>(d), SRC_NONE, 0);
        loc_src[i] = SRC_REG;
        loc_idx[i] = static_cast<uint32_t>(d);
        if (last_use[i] < 0) busy[d] = false;
        break;
      }
      case GE_SIGMOID:
      case GE_TANH:
      case GE_GELU:
      case GE_SILU:
      case GE_HARDSWISH: {
        // the operand is read from wherever it lives; its register is
        // reused when this is its last use
        const uint32_t op = nd.op == GE_SIGMOID ? OP_SIGMOID
                            : nd.op == GE_TANH  ? OP_TANH
                            : nd.op == GE_GELU  ? OP_GELU
                            : nd.op == GE_SILU  ? OP_SILU
                                                : OP_HARDSWISH;
        int d = -1;
        if (loc_src[nd.a] == SRC_REG && last_use[nd.a] == i) {
          d = static_cast<int>(loc_idx[nd.a]);
        } else {
          for (int r = 0; r < kRegs; ++r)
            if (!busy[r]) {
              d = r;
              break;
            }
          if (d < 0) {
            R.status = GE_ERR_UNSUPPORTED;
            return R;
          }
          busy[d] = true;
          if (d + 1 > max_regs) max_regs = d + 1;
        }
        P.ins[P.n_ins++] = pack_ins(op, static_cast<uint32_t>(d), loc_src[nd.a], loc_idx[nd.a]);
        loc_src[i] = SRC_REG;
        loc_idx[i] = static_cast<uint32_t>(d);
        if (last_use[i] < 0) busy[d] = false;
        break;
      }
      case GE_STORE:
        P.ins[P.n_ins++] =
            pack_ins(OP_STORE, static_cast<uint32_t>(nd.slot), loc_src[nd.a], loc_idx[nd.a]);
        if (loc_src[nd.a] == SRC_REG && last_use[nd.a] == i) busy[loc_idx[nd.a]] = false;
        break;
      default:
        R.status = GE_ERR_UNSUPPORTED;
        return R;
    }
  }
  P.n_out = dt.n_out;
  for (int o = 0; o < dt.n_out; ++o) P.out_dtype[o] = dt.out[o];
  P.n_regs = max_regs;
  return R;
}

// Same program (instructions and operand types); scalar values are run-time.
__host__ __device__ constexpr bool same_program(const EpiProgram &a, const EpiProgram &b) {
  if (a.n_ins != b.n_ins || a.n_tma_aux != b.n_tma_aux || a.n_bcast != b.n_bcast ||
      a.n_cbcast != b.n_cbcast || a.n_out != b.n_out)
    return false;
  for (int t = 0; t < a.n_cbcast; ++t)
    if (a.cbcast_dtype[t] != b.cbcast_dtype[t]) return false;
  for (int i = 0; i < a.n_ins; ++i)
    if (a.ins[i] != b.ins[i]) return false;
  for (int t = 0; t < a.n_tma_aux; ++t)
    if (a.tma_aux_dtype[t] != b.tma_aux_dtype[t]) return false;
  for (int t = 0; t < a.n_bcast; ++t)
    if (a.bcast_dtype[t] != b.bcast_dtype[t]) return false;
  for (int o = 0; o < a.n_out; ++o)
    if (a.out_dtype[o] != b.out_dtype[o]) return false;
  return true;
}

}  // namespace ge
