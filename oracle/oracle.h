/*
 * oracle.h -- plain fp64 CPU oracle for a batched dense GEMM whose result is
 * passed through an elementwise epilogue DAG.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this code: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (the plain definition, no blocking or fusion):
 *
 *   accum[l,i,j] = sum_{k=0..K-1} A[l,i,k] * B[l,k,j]          in fp64, k in order
 *
 * "CUTLASS Operator API: Custom epilogue fusions for GEMMs", section
 * "Defining an epilogue via a Python function": the epilogue receives the
 * accumulator `accum` (the GEMM result before the epilogue) and further tensor
 * or scalar operands, applies elementwise operations written in single
 * assignment form, and returns one or more outputs, one of them named D.
 * Section "How the epilogue fusion API works" (figure "Intermediate DAG
 * representation") draws that function as a DAG of AccFetch, Load, compute and
 * Store nodes.  The oracle evaluates such a DAG node by node, for every output
 * element, in fp64:
 *
 *   ORC_ACCUM      -> accum[l,i,j]
 *   ORC_LOAD  s    -> aux_s[l,i,j]            (aux tensor of shape (L,M,N))
 *   ORC_BCAST s    -> aux_s[j]                (row broadcast: shape (N,), the same
 *                                              vector for every row i and batch l;
 *                                              same page, "Row and column broadcasts")
 *   ORC_SCALAR s   -> scalar_s
 *   ORC_MUL a b    -> v[a] * v[b]
 *   ORC_ADD a b    -> v[a] + v[b]
 *   ORC_RELU a     -> v[a] > 0 ? v[a] : +0    ("Custom Epilogue Example",
 *                                              section "Activation Functions")
 *   ORC_SUB a b    -> v[a] - v[b]             (same page as the DAG, section
 *   ORC_DIV a b    -> v[a] / v[b]              "Defining an epilogue via a Python
 *   ORC_MIN a b    -> v[b] < v[a] ? v[b] : v[a]  function": tensor-tensor and
 *   ORC_MAX a b    -> v[b] > v[a] ? v[b] : v[a]  scalar add/sub/mul/div, binary
 *                                              minimum and maximum)
 *   ORC_COLBCAST s -> aux_s[i]                (column broadcast: shape (M,) or
 *                                              (M, 1), the same for every column
 *                                              j and batch l)
 *   activations of v[a] (the legacy Python interface's activation registry:
 *   gelu, hardswish, identity, leaky_relu, relu, sigmoid, silu, tanh; the
 *   operator API's "Predefined elementwise activation functions"):
 *   ORC_SIGMOID    -> 1 / (1 + exp(-x))
 *   ORC_TANH       -> tanh(x)
 *   ORC_GELU       -> x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2)))
 *   ORC_SILU       -> x * sigmoid(x) = x / (1 + exp(-x))
 *   ORC_HARDSWISH  -> x * min(max(x + 3, 0), 6) / 6
 *   ORC_LEAKY_RELU a b -> v[a] > 0 ? v[a] : v[b] * v[a]   (v[b]: the slope)
 *   ORC_STORE a s  -> out_s[l,i,j] = round_to_nearest_even(type_s, v[a])
 *
 * Only a store rounds; every intermediate value stays in fp64 (the pages run
 * the epilogue in fp32: "Custom Epilogue Example", section "Running the
 * Example", --epi_dtype Float32; fp64 is the exact-arithmetic stand-in).  The
 * rounding to fp16 / bf16 is done directly from fp64, written from the
 * IEEE 754 binary16 definition and the bfloat16 definition (1 sign bit,
 * 8 exponent bits, 7 fraction bits), with ties to even and overflow to inf.
 *
 * Parity pins: every function here is checked by tests that do not call it to
 * produce their expected values (exhaustive codec checks, exact integer closed
 * forms, exact rational brute force, a hand-worked example, special cases).
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2 };

/* DAG node kinds */
enum {
  ORC_ACCUM = 0,
  ORC_LOAD = 1,
  ORC_SCALAR = 2,
  ORC_BCAST = 3,
  ORC_MUL = 4,
  ORC_ADD = 5,
  ORC_RELU = 6,
  ORC_STORE = 7,
  ORC_SUB = 8,
  ORC_DIV = 9,
  ORC_MIN = 10,
  ORC_MAX = 11,
  ORC_COLBCAST = 12,
  ORC_SIGMOID = 13,
  ORC_TANH = 14,
  ORC_GELU = 15,
  ORC_SILU = 16,
  ORC_HARDSWISH = 17,
  ORC_LEAKY_RELU = 18
};

typedef struct {
  int32_t op;   /* ORC_* node kind */
  int32_t a;    /* first operand: index of an earlier node */
  int32_t b;    /* second operand (MUL, ADD) */
  int32_t slot; /* aux slot (LOAD, BCAST), scalar slot (SCALAR), out slot (STORE) */
} orc_node;

/* return codes of orc_gemm_epilogue */
enum {
  ORC_OK = 0,
  ORC_BAD_ARGS = -1, /* NULL pointer, non-positive size, unknown type */
  ORC_BAD_DAG = -2,  /* operand not an earlier value node, slot out of range */
  ORC_NO_MEM = -3
};

/* Scalar codecs (exported so the tests can pin them exhaustively). */
double orc_f16_to_f64(uint16_t h);
double orc_bf16_to_f64(uint16_t h);
uint16_t orc_f64_to_f16(double x);
uint16_t orc_f64_to_bf16(double x);

/*
 * Evaluate the GEMM and the epilogue DAG for a list of output rows.
 *
 *  L, M, N, K     problem sizes (all > 0)
 *  ab_type        ORC_F16 or ORC_BF16: element type of A and B (raw 16-bit codes)
 *  A              L*M*K codes, row-major (l, i, k)
 *  B              L*K*N codes, row-major (l, k, j)
 *  n_aux          number of aux slots; aux_type[s] in {F16, BF16, F32}
 *  aux[s]         LOAD slots: L*M*N elements row-major (l, i, j);
 *                 BCAST slots: N elements; COLBCAST slots: M elements;
 *                 raw codes for F16/BF16, float for F32
 *  n_scalar       number of scalars; scalars[s] as double
 *  n_nodes,nodes  the DAG in topological (single assignment) order
 *  n_out          number of outputs; out_type[o] in {F16, BF16, F32}
 *  n_rows, rows   the rows to compute, each r = l*M + i in [0, L*M);
 *                 rows == NULL means all L*M rows in order (n_rows ignored)
 *  outs[o]        n_rows*N elements, row-major (row position in the list, j):
 *                 uint16 codes for F16/BF16, float for F32
 *  pre[o]         optional (array or entries may be NULL): n_rows*N doubles,
 *                 the fp64 value each store rounded
 *  n_threads      worker threads (<= 0: all online processors)
 */
int orc_gemm_epilogue(int64_t L, int64_t M, int64_t N, int64_t K, int32_t ab_type,
                      const uint16_t *A, const uint16_t *B, int32_t n_aux,
                      const int32_t *aux_type, const void *const *aux, int32_t n_scalar,
                      const double *scalars, int32_t n_nodes, const orc_node *nodes,
                      int32_t n_out, const int32_t *out_type, void *const *outs,
                      double *const *pre, int64_t n_rows, const int64_t *rows,
                      int32_t n_threads);

/* Plain fp64 accumulator rows only: acc[r][j] for the listed rows (same
 * conventions as above). */
int orc_gemm_accum(int64_t L, int64_t M, int64_t N, int64_t K, int32_t ab_type,
                   const uint16_t *A, const uint16_t *B, double *acc, int64_t n_rows,
                   const int64_t *rows, int32_t n_threads);

#ifdef __cplusplus
}
#endif

#endif /* ORACLE_H */
