/*
 * gemm_epi.h -- C ABI of libgemm_epi.so: a batched dense GEMM on one GB300
 * (sm_103a) whose elementwise epilogue is fused into the same kernel.
 *
 *   accum[l] = A[l] @ B[l]                         fp16/bf16 operands, fp32 accumulate
 *   outs     = epilogue DAG (accum, aux tensors, row-broadcast vectors, scalars)
 *
 * What the operation is: "CUTLASS Operator API: Custom epilogue fusions for
 * GEMMs", sections "Custom epilogue fusions for GEMMs" (a GEMM whose result,
 * accum, is transformed by a user epilogue before it is stored; outputs D and
 * Aux, cells [2]-[5]) and "How the epilogue fusion API works" (the epilogue
 * as a DAG of AccFetch, Load, compute and Store nodes).  The node set here is
 * that figure's plus Scalar, row and column Broadcast (section "Row and
 * column broadcasts"), subtraction, division, minimum and maximum, ReLU
 * (section "Defining an epilogue via a Python function": supported
 * operations; "Custom Epilogue Example", section "Activation Functions") and
 * the activation registry of the legacy interface (sigmoid, tanh, GELU,
 * SiLU, hardswish, leaky ReLU).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Layouts are row-major and packed (other storage orders: ge_options):
 *      A      (L, M, K)   K contiguous
 *      B      (L, K, N)   N contiguous
 *      aux tensors and outputs (L, M, N), N contiguous
 *      row-broadcast vectors (N,), one vector for every row of every batch;
 *      column-broadcast vectors (M,) (the pages' (M, 1)), one value per row,
 *      the same for every column and every batch.
 *  * Every device pointer must be 16-byte aligned and every row of a 2-D/3-D
 *    operand must be a multiple of 16 bytes long ("Custom Epilogue Example",
 *    section "Constraints": contiguous dimensions 16-byte aligned).
 *  * The caller owns all device memory (A, B, aux, outputs, the unfused
 *    workspace).  A batched plan owns only host state; creating one
 *    allocates no device memory (grouped plans own their problem tables).
 *    Plans are not thread-safe: use one plan per host thread.
 *  * `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Runs are asynchronous on that stream; nothing synchronises.
 *  * The epilogue runs in fp32: every intermediate stays fp32 and only a
 *    store rounds (round to nearest even) to its output type ("Custom
 *    Epilogue Example", "Running the Example": --acc_dtype Float32,
 *    --epi_dtype Float32).  ReLU returns +0 for inputs <= 0.
 *  * Results are bit-for-bit repeatable for a given plan on a given device.
 *    The order of the sum over K belongs to the plan (tile shape, grid,
 *    and a tile's place in the schedule: a CTA walks K upwards on its even
 *    tiles and downwards on its odd ones), so two plans that differ in those
 *    may round non-integer results differently, within fp32 summation error;
 *    the epilogue warp count, the last-wave split and the fused/unfused
 *    choice never change the result.
 *  * Return values are GE_* status codes; gemm_epi_status_string names them.
 */
#ifndef GEMM_EPI_H
#define GEMM_EPI_H

#ifdef __CUDACC_RTC__
/* the library compiling its own kernels at run time: no C library headers */
typedef signed char int8_t;
typedef short int16_t;
typedef int int32_t;
typedef long long int64_t;
typedef unsigned char uint8_t;
typedef unsigned short uint16_t;
typedef unsigned int uint32_t;
typedef unsigned long long uint64_t;
#else
#include <stddef.h>
#include <stdint.h>
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define GE_MAX_NODES 16   /* nodes in one epilogue DAG */
#define GE_MAX_AUX 8      /* aux slots (Load tensors and Broadcast vectors) */
#define GE_MAX_TMA_AUX 4  /* of which Load tensors */
#define GE_MAX_OUT 4      /* output slots */
#define GE_MAX_SCALARS 16 /* scalar slots */

/* element types */
typedef enum { GE_F16 = 0, GE_BF16 = 1, GE_F32 = 2 } ge_dtype;

/* DAG node kinds.  `a`, `b` name earlier nodes; `slot` picks the operand. */
typedef enum {
  GE_ACCFETCH = 0,  /* the fp32 accumulator accum[l,i,j]                     */
  GE_LOAD = 1,      /* aux slot `slot`, an (L,M,N) tensor: aux[l,i,j]        */
  GE_SCALAR = 2,    /* scalar slot `slot`                                    */
  GE_BROADCAST = 3, /* aux slot `slot`, an (N,) row vector: aux[j]           */
  GE_MUL = 4,       /* v[a] * v[b]                                           */
  GE_ADD = 5,       /* v[a] + v[b]                                           */
  GE_RELU = 6,      /* v[a] > 0 ? v[a] : +0                                  */
  GE_STORE = 7,     /* out slot `slot` = round(v[a]); slot 0 is D            */
  GE_SUB = 8,       /* v[a] - v[b]                                           */
  GE_DIV = 9,       /* v[a] / v[b]  (fp32, correctly rounded)                */
  GE_MIN = 10,      /* min(v[a], v[b])                                       */
  GE_MAX = 11,      /* max(v[a], v[b])                                       */
  GE_COL_BROADCAST = 12, /* aux slot `slot`, an (M,) column vector: aux[i]   */
  /* Activations of the legacy interface's registry (Python examples
   * walkthrough, epilogue notebook), evaluated in fp32 with the CUDA math
   * library's expf / tanhf / erfcf (not bit-reproducible against another
   * libm: compare within a tolerance).                                      */
  GE_SIGMOID = 13,    /* 1 / (1 + exp(-v[a]))                                */
  GE_TANH = 14,       /* tanh(v[a])                                          */
  GE_GELU = 15,       /* v[a]/2 * (1 + erf(v[a] / sqrt(2)))  (exact GELU)     */
  GE_SILU = 16,       /* v[a] / (1 + exp(-v[a]))                             */
  GE_HARDSWISH = 17,  /* v[a] * min(max(v[a] + 3, 0), 6) / 6                 */
  GE_LEAKY_RELU = 18  /* v[a] > 0 ? v[a] : v[b] * v[a]  (v[b]: the slope)    */
} ge_op;

typedef struct {
  int32_t op;   /* ge_op */
  int32_t a;    /* first operand (node index) */
  int32_t b;    /* second operand of the two-operand nodes */
  int32_t slot; /* aux / scalar / output slot */
} ge_node;

/* The epilogue function as a DAG in single assignment, topological order:
 * every operand refers to an earlier node, every output slot is stored
 * exactly once (the pages' SSA rule: a variable is assigned once). */
typedef struct {
  int32_t n;
  ge_node node[GE_MAX_NODES];
} ge_dag;

typedef struct {
  int32_t ab;                   /* GE_F16 or GE_BF16: type of A and B          */
  int32_t acc;                  /* must be GE_F32                              */
  int32_t n_aux;                /* aux slots used (<= GE_MAX_AUX)              */
  int32_t n_scalar;             /* scalar slots (<= GE_MAX_SCALARS)            */
  int32_t n_out;                /* output slots (1..GE_MAX_OUT); out[0] is D   */
  int32_t aux[GE_MAX_AUX];      /* type of each aux slot                       */
  int32_t out[GE_MAX_OUT];      /* type of each output slot                    */
} ge_dtypes;

/* Storage order of a matrix operand ("Custom Epilogue Example", step
 * "Define tensor arguments": a_major, b_major, cd_major). */
typedef enum { GE_ROW_MAJOR = 0, GE_COL_MAJOR = 1 } ge_major;

/* Optional knobs; zero-initialise for automatic choices and row-major data. */
typedef struct {
  int32_t cta_group;    /* 0 auto, 1 = one CTA per MMA tile, 2 = CTA pair (2x1 cluster) */
  int32_t tile_n;       /* 0 auto, else the MMA N: 64, 128 or 256                       */
  int32_t stages;       /* 0 auto (as many as fit), else 2..8 shared-memory stages      */
  int32_t max_ctas;     /* 0 = one CTA per SM, else a cap on the persistent grid        */
  int32_t raster_group; /* 0 auto, else M tiles per raster group (L2 reuse of B); auto:
                           all M tiles when there are at most 16, else 12 (grouped: 8) */
  int32_t timeout_ms;   /* 0 = 1000; bound on every device-side wait                    */
  uint32_t debug_flags; /* 0; GE_DEBUG_* below, for tests only                          */
  int32_t cluster_n;    /* 0 or 1 (one CTA, or one CTA pair, per cluster); any other
                           value is GE_ERR_UNSUPPORTED.  Every TMA load lands in the
                           issuing CTA's own shared memory: no cluster multicast.     */
  /* Storage order, packed in every case (GE_ERR_INVALID for other values):
   *   a_major   GE_ROW_MAJOR: A is (L,M,K), K contiguous ("K-major");
   *             GE_COL_MAJOR: stored (L,K,M), M contiguous ("M-major")
   *   b_major   GE_ROW_MAJOR: B is (L,K,N), N contiguous ("N-major");
   *             GE_COL_MAJOR: stored (L,N,K), K contiguous ("K-major")
   *   cd_major  every Load tensor and every output, alike (the pages'
   *             same-major rule for epilogue tensors): GE_ROW_MAJOR (L,M,N),
   *             N contiguous; GE_COL_MAJOR stored (L,N,M), M contiguous.
   *             Row and column vectors are unaffected.
   * The contiguous dimension of each tensor must be whole 16-byte units
   * (GE_ERR_MISALIGNED). */
  int32_t a_major;
  int32_t b_major;
  int32_t cd_major;
  /* 0 auto, else the epilogue warps per CTA: 4 (one per accumulator lane
   * quarter) or 8 (two per quarter, each taking every other 32-column
   * step).  Auto is 8, except 4 for the interpreter of programs with more
   * than four live values.  Results are identical either way;
   * GE_ERR_INVALID otherwise.                                              */
  int32_t epi_warps;
  /* 0 (default): an epilogue outside the built-in set gets a fused kernel
   * compiled for its program when the plan is made (the built-in kernels'
   * straight-line code; results identical to the interpreter's), if the CUDA
   * runtime compiler (libnvrtc) can be loaded and the library's sources are
   * next to it; otherwise, or if that compilation fails, the interpreter.
   * A compiled kernel is kept for the life of the process; compiling takes
   * about half a second.  -1: always the interpreter.  The unfused path
   * always interprets.                                                    */
  int32_t specialize;
  /* 0 (default): batched runs are launched with programmatic stream
   * serialization, so a run may start while the previous kernel on its
   * stream is finishing: its set-up (barriers, TMEM allocation) overlaps
   * that kernel's tail, and it reads no input and writes no output before
   * that kernel has completed and its memory is visible.  A run also lets
   * the next launch on the stream be scheduled once it has issued its last
   * operand copy.  Nonzero: plain launches.  A grouped run overlaps only
   * when it reuses its problem table from a run on the same stream (no
   * table copy and no cross-stream wait precede it).                        */
  int32_t no_pdl;
} ge_options;

/* Test hook: the producer never loads the first k-block, so the MMA warp's
 * wait on it runs out after timeout_ms and the run reports GE_ERR_TIMEOUT.
 * Nothing faults or hangs: every wait in the kernel is bounded. */
#define GE_DEBUG_SKIP_FIRST_LOAD 1u

/* Run the epilogue through the general interpreter even when the DAG matches
 * a built-in (precompiled, straight-line) epilogue.  Results are identical;
 * used to test that the two executors agree. */
#define GE_DEBUG_FORCE_INTERPRETER 2u

/* Keep every tile of a batched launch full width.  By default, when the last
 * wave of tiles would leave at least half of the CTAs (pairs) idle, each of
 * its tiles is split into two half-width tiles; results are identical either
 * way (each output element's sum runs over K in the same order), so tests
 * compare the two schedules. */
#define GE_DEBUG_NO_TAIL_SPLIT 4u

/* What a plan chose (for logs, tests and the benchmark). */
typedef struct {
  int32_t cta_group, tile_m, tile_n, tile_k;  /* tile_m/tile_n: output tile of one MMA */
  int32_t stages, epi_chunk, aux_stages;
  int32_t grid, num_tiles, smem_bytes;
  int32_t n_instr, n_regs;                    /* compiled epilogue program             */
  int32_t num_sms;
  int32_t epi_variant;                        /* built-in epilogue used; -1, -2: interpreter
                                                 (4 / 8 program registers); -3: compiled for
                                                 this program when the plan was made        */
  int32_t cluster_n;                          /* always 1: no operand sharing between pairs */
  int32_t epi_warps;                          /* epilogue warps per CTA (4 or 8)         */
  int32_t raster_group;                       /* M tiles per raster group (batched: the
                                                 group in effect, at most the M tiles)    */
} ge_plan_info;

typedef struct gemm_epi_plan gemm_epi_plan;

/* status codes */
enum {
  GE_OK = 0,
  GE_ERR_NO_ACCUM = 1,    /* DAG has no GE_ACCFETCH ("accum must be an input to the epilogue") */
  GE_ERR_NO_D = 2,        /* no GE_STORE to slot 0 ("Output node D is not found")               */
  GE_ERR_SSA = 3,         /* operand is not an earlier value node, or a slot is stored twice   */
  GE_ERR_MISSING_ARG = 4, /* slot beyond n_aux/n_scalar/n_out, or a NULL operand at run time   */
  GE_ERR_UNSUPPORTED = 5, /* unknown op or type, too many nodes/slots, program too large       */
  GE_ERR_MISALIGNED = 6,  /* pointer or row length not a multiple of 16 bytes                  */
  GE_ERR_ARCH = 7,        /* no compute-capability 10.3 device current                         */
  GE_ERR_SHAPE = 8,       /* L, M, N or K <= 0 or too large                                    */
  GE_ERR_TIMEOUT = 9,     /* a device-side wait ran out (read with gemm_epi_last_error)        */
  GE_ERR_CUDA = 10,       /* a CUDA runtime / driver call failed                               */
  GE_ERR_INVALID = 11,    /* NULL plan or struct, bad option, output slot never stored         */
  GE_ERR_SMEM = 12,       /* the requested tile/stages do not fit in shared memory             */
  GE_ERR_WORKSPACE = 13   /* unfused workspace missing, misaligned or too small                */
};

/*
 * Validate the epilogue and the problem and build a plan.  Host only: checks
 * the DAG and the types first (no device needed for those errors), then the
 * current device (compute capability 10.3) and the shared-memory budget,
 * then compiles the DAG into the kernel's epilogue program and picks the
 * tile, the stage count and the persistent grid.
 *   plan   out: the new plan (NULL on failure)
 *   L,M,N,K   batch count and GEMM sizes, all > 0
 * Errors: GE_ERR_INVALID, _SHAPE, _UNSUPPORTED, _NO_ACCUM, _NO_D, _SSA,
 * _MISSING_ARG, _MISALIGNED (row lengths), _ARCH, _SMEM, _CUDA.
 */
int gemm_epi_plan_create(gemm_epi_plan **plan, int64_t L, int64_t M, int64_t N, int64_t K,
                         const ge_dtypes *dtypes, const ge_dag *dag);

/* Same with tuning options (opts may be NULL). */
int gemm_epi_plan_create_ex(gemm_epi_plan **plan, int64_t L, int64_t M, int64_t N, int64_t K,
                            const ge_dtypes *dtypes, const ge_dag *dag, const ge_options *opts);

/*
 * Host-only check of a DAG against its types, with the same codes as
 * gemm_epi_plan_create; touches no device.
 */
int gemm_epi_validate(const ge_dtypes *dtypes, const ge_dag *dag);

/*
 * Run the fused GEMM + epilogue: one persistent kernel launch on `stream`.
 *   A, B      device pointers (layouts above)
 *   aux       n_aux device pointers; entries for slots the DAG never reads may be NULL
 *   scalars   n_scalar host floats (read during the call; may be NULL if n_scalar == 0)
 *   outs      n_out device pointers, each (L,M,N) of its output type
 * Errors: GE_ERR_INVALID (also for a grouped plan), _MISSING_ARG,
 * _MISALIGNED, _CUDA (launch failed).  A device-side timeout is reported
 * later by gemm_epi_last_error.  Tensor maps are encoded on the host when
 * a pointer differs from the previous run's; a run with the same pointers
 * only launches, so it can be captured into a CUDA graph.  The unfused entry points below reject
 * grouped plans the same way.
 */
int gemm_epi_run(gemm_epi_plan *plan, const void *A, const void *B, const void *const *aux,
                 const float *scalars, void *const *outs, void *stream);

/* Bytes of fp32 workspace gemm_epi_run_unfused needs: L*M*N*4. */
size_t gemm_epi_unfused_workspace_bytes(const gemm_epi_plan *plan);

/*
 * The unfused comparison path ("Custom Epilogue Example", section
 * "Overview": the GEMM in one kernel, the elementwise work in another).
 * Launch 1: the same GEMM kernel stores the fp32 accumulator into
 * `workspace`; launch 2: a vectorised elementwise kernel reads it back with
 * the aux operands and evaluates the same epilogue program, so results are
 * bit-identical to gemm_epi_run.
 *   workspace        caller-owned device buffer of >= gemm_epi_unfused_workspace_bytes;
 *                    it receives accum in the epilogue tensors' storage order
 *                    ((L,M,N), or (L,N,M) with cd_major GE_COL_MAJOR)
 * Errors: as gemm_epi_run, plus GE_ERR_WORKSPACE.
 */
int gemm_epi_run_unfused(gemm_epi_plan *plan, const void *A, const void *B,
                         const void *const *aux, const float *scalars, void *const *outs,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * Allocation-free variant of gemm_epi_run_unfused.  No counterpart on the
 * pages: it exists for callers that cannot allocate device memory — code that
 * runs where a cudaMalloc is not allowed or not wanted (inside an allocator or
 * memory-pool callback, in a host application that reserves every byte of
 * device memory up front and hands out nothing else, or in a deployment that
 * forbids allocation after start-up) and so cannot provide the fp32
 * workspace the unfused path needs.
 *
 * Instead of a caller buffer it uses one workspace compiled into the library:
 * a device array of GE_NOALLOC_SCRATCH_BYTES that every GPU loading this
 * library holds until the process exits.  The caller still passes A, B, aux,
 * scalars and outputs exactly as for gemm_epi_run_unfused, and the results are
 * the same bits.  The call itself allocates nothing.
 *
 *  * Problems needing more than GE_NOALLOC_SCRATCH_BYTES of workspace
 *    (L*M*N*4 bytes) are rejected with GE_ERR_WORKSPACE before any launch.
 *  * The first call on a device looks up that device's address of the array
 *    (cudaGetSymbolAddress, with that device current); make the first call on
 *    each device before any stream capture.  The address is kept for the
 *    life of the process: after a cudaDeviceReset it, like every plan made
 *    before the reset, is no longer valid, so do not use this library on
 *    that device again in the same process.
 *  * All calls share the one array and it keeps whatever the last call left
 *    in it.  Nothing in it needs to start at zero: the GEMM overwrites every
 *    element it later reads.  Calls whose work overlaps on the GPU (different
 *    streams, or different host threads, same device) race on the array: the
 *    caller must order them.
 * Errors: as gemm_epi_run_unfused, GE_ERR_WORKSPACE for oversized problems,
 * GE_ERR_CUDA if the set-up lookup fails.
 */
#define GE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int gemm_epi_run_unfused_noalloc(gemm_epi_plan *plan, const void *A, const void *B,
                                 const void *const *aux, const float *scalars, void *const *outs,
                                 void *stream);

/*
 * Grouped GEMM with a fused epilogue ("Grouped GEMM" in example three of the
 * CUTLASS Python interface walkthrough; "Combine custom epilogues with
 * grouped operations" under Next Steps of "Custom Epilogue Example"):
 * n_problems independent problems of different sizes,
 *   outs_g = epilogue(A_g @ B_g, aux_g, scalars),  g = 0 .. n_problems-1,
 * with one DAG, one set of types and one set of scalars for all of them,
 * computed by a single persistent launch over the tiles of every problem.
 * Each problem is laid out like one batch of gemm_epi_run: A_g (M,K), B_g
 * (K,N), Load tensors and outputs (M,N), row vectors (N,), column vectors
 * (M,), row-major and packed; the same 16-byte rules apply per problem.
 */
typedef struct {
  int64_t M, N, K; /* all > 0 */
} ge_problem;

#define GE_MAX_GROUPS 4096 /* problems in one grouped plan */

/*
 * Build a grouped plan.  Validation as gemm_epi_plan_create_ex, per problem;
 * opts may be NULL.  The plan allocates its tables: four problem tables
 * in device memory and their pinned host staging (1.5 KiB per problem each)
 * and the launch's tile order (16 bytes per output tile), which it uploads
 * once with a synchronous copy (GE_ERR_CUDA if any of that fails).  Errors:
 * those of gemm_epi_plan_create_ex, and GE_ERR_SHAPE when n_problems is
 * outside 1..GE_MAX_GROUPS or the problems have more than 2^24 output tiles.
 */
int gemm_epi_grouped_plan_create(gemm_epi_plan **plan, int32_t n_problems,
                                 const ge_problem *problems, const ge_dtypes *dtypes,
                                 const ge_dag *dag, const ge_options *opts);

/*
 * Run a grouped plan on `stream`.  Host arrays of device pointers:
 *   A, B     n_problems entries each
 *   aux      n_problems * n_aux entries, problem-major: aux[g*n_aux + slot]
 *            (NULL allowed when the DAG reads no aux slot)
 *   outs     n_problems * n_out entries: outs[g*n_out + slot]
 *   scalars  host fp32, n_scalar values shared by every problem
 * The problem table (tensor maps and vector pointers) is built on the host
 * and copied to the device with the launch.  When every pointer equals the
 * previous run's, that table is reused and nothing is copied; otherwise the
 * next of four tables is rebuilt, which first waits (on the host) for the
 * run that last used that table to finish.  Errors: GE_ERR_INVALID (NULL or
 * not a grouped plan), GE_ERR_MISSING_ARG, GE_ERR_MISALIGNED, GE_ERR_CUDA.
 */
int gemm_epi_grouped_run(gemm_epi_plan *plan, const void *const *A, const void *const *B,
                         const void *const *aux, const float *scalars, void *const *outs,
                         void *stream);

/* Free a plan (NULL is ignored).  Does not synchronise, except that a
 * grouped plan first waits for the runs still reading its tables. */
void gemm_epi_plan_destroy(gemm_epi_plan *plan);

/* Fill `info` with the plan's choices.  Errors: GE_ERR_INVALID. */
int gemm_epi_plan_info(const gemm_epi_plan *plan, ge_plan_info *info);

/* Static name of a status code ("GE_OK", ...); never NULL. */
const char *gemm_epi_status_string(int status);

/*
 * Read and clear the sticky device-side status of the current device:
 * GE_OK, or GE_ERR_TIMEOUT when some wait in a kernel of this library gave
 * up (the kernel then stopped early and its outputs are undefined).  The
 * status word is shared by all plans on a device.  Call it after the runs
 * of interest have completed (e.g. after synchronising their stream); it
 * performs a synchronous device-to-host copy.  plan may be NULL.
 */
int gemm_epi_last_error(gemm_epi_plan *plan);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_EPI_H */
