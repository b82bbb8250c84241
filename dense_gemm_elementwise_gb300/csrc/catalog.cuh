// catalog.cuh -- built-in epilogues with precompiled straight-line kernels.
//
// Each entry is an ordinary epilogue DAG plus operand types.  At build time
// compile_program() turns it into the same instruction list the plan
// compiler produces for a user DAG; the kernels for an entry evaluate that
// list with every dispatch resolved at compile time.  A plan whose compiled
// program equals an entry's (same instructions, same operand types; scalar
// values are free) uses that entry's kernels, any other DAG the interpreter.
// The entries cover the common fused epilogues of the pages: storing the
// accumulator, linear combinations with an aux tensor, ReLU, row-broadcast
// bias, auxiliary outputs, a squared second output and GELU over a linear
// combination.
#pragma once

#include "program.cuh"

namespace ge {
namespace catalog {

struct Entry {
  const char *name;
  ge_dtypes dt;
  ge_dag dag;
};

constexpr ge_node nd(int op, int a = 0, int b = 0, int slot = 0) { return ge_node{op, a, b, slot}; }

constexpr ge_dtypes types(int n_aux, int aux0, int aux1, int n_scalar, int n_out, int out0, int out1,
                          int aux2 = 0) {
  ge_dtypes d{};
  d.ab = GE_F16;  // A/B type is a kernel parameter, not part of the program
  d.acc = GE_F32;
  d.n_aux = n_aux;
  d.n_scalar = n_scalar;
  d.n_out = n_out;
  d.aux[0] = aux0;
  d.aux[1] = aux1;
  d.aux[2] = aux2;
  d.out[0] = out0;
  d.out[1] = out1;
  return d;
}

// accum stored as-is (also the first kernel of the unfused path)
constexpr ge_dag dag_store_accum() { return ge_dag{2, {nd(GE_ACCFETCH), nd(GE_STORE, 0, 0, 0)}}; }

// Aux = alpha*accum + beta*C ; D = extra_scalar*Aux
constexpr ge_dag dag_aux_scaled() {
  return ge_dag{11,
                {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 1, 0), nd(GE_LOAD, 0, 0, 0),
                 nd(GE_SCALAR, 0, 0, 1), nd(GE_MUL, 4, 3), nd(GE_ADD, 2, 5), nd(GE_SCALAR, 0, 0, 2),
                 nd(GE_MUL, 7, 6), nd(GE_STORE, 8, 0, 0), nd(GE_STORE, 6, 0, 1)}};
}

// D = alpha*accum + beta*C, optionally through ReLU
constexpr ge_dag dag_linear(bool relu) {
  ge_dag g{7,
           {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 0, 1), nd(GE_LOAD, 0, 0, 0),
            nd(GE_SCALAR, 0, 0, 1), nd(GE_MUL, 3, 4), nd(GE_ADD, 2, 5)}};
  if (relu) {
    g.node[7] = nd(GE_RELU, 6);
    g.node[8] = nd(GE_STORE, 7, 0, 0);
    g.n = 9;
  } else {
    g.node[7] = nd(GE_STORE, 6, 0, 0);
    g.n = 8;
  }
  return g;
}

// Y = accum ; D = alpha*accum + beta*C + x_factor*X
constexpr ge_dag dag_alpha_beta_x() {
  return ge_dag{13,
                {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 0, 1), nd(GE_LOAD, 0, 0, 0),
                 nd(GE_SCALAR, 0, 0, 1), nd(GE_MUL, 3, 4), nd(GE_ADD, 2, 5), nd(GE_LOAD, 0, 0, 1),
                 nd(GE_SCALAR, 0, 0, 2), nd(GE_MUL, 7, 8), nd(GE_ADD, 6, 9), nd(GE_STORE, 10, 0, 0),
                 nd(GE_STORE, 0, 0, 1)}};
}

// D = relu(alpha*accum + beta*C + bias) ; E = D*D
constexpr ge_dag dag_bias_relu_square() {
  return ge_dag{13,
                {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 1, 0), nd(GE_SCALAR, 0, 0, 1),
                 nd(GE_LOAD, 0, 0, 0), nd(GE_MUL, 3, 4), nd(GE_ADD, 2, 5), nd(GE_BROADCAST, 0, 0, 1),
                 nd(GE_ADD, 6, 7), nd(GE_RELU, 8), nd(GE_MUL, 9, 9), nd(GE_STORE, 9, 0, 0),
                 nd(GE_STORE, 10, 0, 1)}};
}

// D = alpha*accum + bias
constexpr ge_dag dag_row_bias() {
  return ge_dag{6,
                {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 0, 1), nd(GE_BROADCAST, 0, 0, 0),
                 nd(GE_ADD, 2, 3), nd(GE_STORE, 4, 0, 0)}};
}

// D = alpha*accum + row_bias + col_bias
constexpr ge_dag dag_row_col_bias() {
  return ge_dag{8,
                {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 0, 1), nd(GE_BROADCAST, 0, 0, 0),
                 nd(GE_ADD, 2, 3), nd(GE_COL_BROADCAST, 0, 0, 1), nd(GE_ADD, 4, 5),
                 nd(GE_STORE, 6, 0, 0)}};
}

// D = gelu(alpha*accum + C)
constexpr ge_dag dag_linear_gelu() {
  return ge_dag{7,
                {nd(GE_ACCFETCH), nd(GE_SCALAR, 0, 0, 0), nd(GE_MUL, 0, 1), nd(GE_LOAD, 0, 0, 0),
                 nd(GE_ADD, 2, 3), nd(GE_GELU, 4), nd(GE_STORE, 5, 0, 0)}};
}

// D = gelu((accum + bias)*scale + c + tanh(x))
constexpr ge_dag dag_complex_gelu_tanh() {
  return ge_dag{12,
                {nd(GE_ACCFETCH), nd(GE_BROADCAST, 0, 0, 2), nd(GE_ADD, 0, 1), nd(GE_SCALAR, 0, 0, 0),
                 nd(GE_MUL, 2, 3), nd(GE_LOAD, 0, 0, 0), nd(GE_ADD, 4, 5), nd(GE_LOAD, 0, 0, 1),
                 nd(GE_TANH, 7), nd(GE_ADD, 6, 8), nd(GE_GELU, 9), nd(GE_STORE, 10, 0, 0)}};
}

constexpr Entry kEntries[] = {
    {"store_accum_f32", types(0, 0, 0, 0, 1, GE_F32, 0), dag_store_accum()},
    {"store_accum_f16", types(0, 0, 0, 0, 1, GE_F16, 0), dag_store_accum()},
    {"store_accum_bf16", types(0, 0, 0, 0, 1, GE_BF16, 0), dag_store_accum()},
    {"aux_scaled_f16", types(1, GE_F16, 0, 3, 2, GE_F16, GE_F16), dag_aux_scaled()},
    {"linear_relu_f16", types(1, GE_F16, 0, 2, 1, GE_F16, 0), dag_linear(true)},
    {"linear_f16", types(1, GE_F16, 0, 2, 1, GE_F16, 0), dag_linear(false)},
    {"alpha_beta_x_f16", types(2, GE_F16, GE_F16, 3, 2, GE_F16, GE_F16), dag_alpha_beta_x()},
    {"bias_relu_square_bf16", types(2, GE_BF16, GE_F32, 2, 2, GE_BF16, GE_BF16),
     dag_bias_relu_square()},
    {"row_bias_f16", types(1, GE_F16, 0, 1, 1, GE_F16, 0), dag_row_bias()},
    {"row_col_bias_f16", types(2, GE_F16, GE_F16, 1, 1, GE_F16, 0), dag_row_col_bias()},
    {"linear_gelu_f16", types(1, GE_F16, 0, 1, 1, GE_F16, 0), dag_linear_gelu()},
    {"complex_gelu_tanh_bf16", types(3, GE_BF16, GE_BF16, 1, 1, GE_BF16, 0, GE_F32),
     dag_complex_gelu_tanh()},
};

constexpr int kCount = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));

template <int K>
struct Prog {
  static constexpr CompileResult R = compile_program(kEntries[K].dt, kEntries[K].dag);
  static_assert(R.status == GE_OK, "catalog entry does not compile");
  static constexpr EpiProgram P = R.prog;
};

}  // namespace catalog
}  // namespace ge
