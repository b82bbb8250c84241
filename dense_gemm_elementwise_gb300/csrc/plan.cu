// plan.cu -- host side of libgemm_epi.so: the C ABI declared in gemm_epi.h.
//
// The DAG rules follow "CUTLASS Operator API: Custom epilogue fusions for
// GEMMs", "Failure examples" (cells [10]-[13]: the accumulator must be an
// input, D must be produced, values are assigned once, every output must be
// provided); the alignment rule follows "Custom Epilogue Example",
// "Constraints" (16-byte aligned contiguous dimensions).
//
//   validate     DAG and type rules (host only, no device needed)
//   compile      ge_dag -> two-address epilogue program (register allocation)
//   configure    tile shape, CTA pairing, stage count, persistent grid
//   run          TMA descriptors (cached per pointer set), one kernel launch
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "catalog.cuh"
#include "common.cuh"
#include "launch.h"
#include "program.cuh"

using namespace ge;

// Device status block: [0] status (GE_OK / GE_ERR_TIMEOUT), [1] wait site,
// [2] block index, [3] unused.  One per device (module global).
__device__ uint32_t g_ge_status[4];

namespace {

int esize(int dt) { return dt == GE_F32 ? 4 : 2; }
bool valid_dtype(int dt) { return dt == GE_F16 || dt == GE_BF16 || dt == GE_F32; }

bool log_enabled() {
  const char *v = std::getenv("GEMM_EPI_LOG");
  return v && *v && *v != '0';
}

// ------------------------------------------------------------- validation --
bool is_value_node(const ge_dag *dag, int ref, int before) {
  return ref >= 0 && ref < before && dag->node[ref].op != GE_STORE;
}

int validate_impl(const ge_dtypes *dt, const ge_dag *dag) {
  if (!dt || !dag) return GE_ERR_INVALID;
  if (dt->ab != GE_F16 && dt->ab != GE_BF16) return GE_ERR_UNSUPPORTED;
  if (dt->acc != GE_F32) return GE_ERR_UNSUPPORTED;
  if (dt->n_aux < 0 || dt->n_aux > GE_MAX_AUX || dt->n_scalar < 0 ||
      dt->n_scalar > GE_MAX_SCALARS || dt->n_out < 1 || dt->n_out > GE_MAX_OUT)
    return GE_ERR_UNSUPPORTED;
  for (int s = 0; s < dt->n_aux; ++s)
    if (!valid_dtype(dt->aux[s])) return GE_ERR_UNSUPPORTED;
  for (int o = 0; o < dt->n_out; ++o)
    if (!valid_dtype(dt->out[o])) return GE_ERR_UNSUPPORTED;
  if (dag->n < 1 || dag->n > GE_MAX_NODES) return GE_ERR_UNSUPPORTED;

  bool has_acc = false;
  int stored[GE_MAX_OUT] = {0};
  int aux_kind[GE_MAX_AUX] = {0};  // 1 Load tensor, 2 row vector, 3 column vector
  for (int i = 0; i < dag->n; ++i) {
    const ge_node &nd = dag->node[i];
    switch (nd.op) {
      case GE_ACCFETCH: has_acc = true; break;
      case GE_LOAD:
      case GE_BROADCAST:
      case GE_COL_BROADCAST: {
        if (nd.slot < 0 || nd.slot >= dt->n_aux) return GE_ERR_MISSING_ARG;
        const int kind = nd.op == GE_LOAD ? 1 : nd.op == GE_BROADCAST ? 2 : 3;
        if (aux_kind[nd.slot] && aux_kind[nd.slot] != kind) return GE_ERR_UNSUPPORTED;
        aux_kind[nd.slot] = kind;
        break;
      }
      case GE_SCALAR:
        if (nd.slot < 0 || nd.slot >= dt->n_scalar) return GE_ERR_MISSING_ARG;
        break;
      case GE_MUL:
      case GE_ADD:
      case GE_SUB:
      case GE_DIV:
      case GE_MIN:
      case GE_MAX:
      case GE_LEAKY_RELU:
        if (!is_value_node(dag, nd.b, i)) return GE_ERR_SSA;
        if (!is_value_node(dag, nd.a, i)) return GE_ERR_SSA;
        break;
      case GE_RELU:
      case GE_SIGMOID:
      case GE_TANH:
      case GE_GELU:
      case GE_SILU:
      case GE_HARDSWISH:
        if (!is_value_node(dag, nd.a, i)) return GE_ERR_SSA;
        break;
      case GE_STORE:
        if (!is_value_node(dag, nd.a, i)) return GE_ERR_SSA;
        if (nd.slot < 0 || nd.slot >= dt->n_out) return GE_ERR_MISSING_ARG;
        if (stored[nd.slot]++) return GE_ERR_SSA;
        break;
      default: return GE_ERR_UNSUPPORTED;
    }
  }
  if (!has_acc) return GE_ERR_NO_ACCUM;
  if (!stored[0]) return GE_ERR_NO_D;
  for (int o = 1; o < dt->n_out; ++o)
    if (!stored[o]) return GE_ERR_INVALID;
  return GE_OK;
}

// catalog entry whose program equals P, or -1
template <int K = 0>
int match_catalog(const EpiProgram &P) {
  if constexpr (K < catalog::kCount) {
    if (same_program(P, catalog::Prog<K>::P)) return K;
    return match_catalog<K + 1>(P);
  } else {
    return -1;
  }
}

// Executor of a compiled program: its catalog entry (k >= 0) unless the
// interpreter is forced, else the interpreter holding 4 (-1) or all kRegs
// (-2) program registers.
int pick_executor(const EpiProgram &P, bool force_interpreter) {
  const int k = force_interpreter ? -1 : match_catalog(P);
  if (k >= 0) return k;
  return P.n_regs > 4 ? -2 : -1;
}

// accumulator-only program of the unfused path's GEMM: out 0 (fp32) = accum
EpiProgram program_store_accum() { return catalog::Prog<0>::P; }

// ---------------------------------------------------------- TMA encoding --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

CUtensorMapDataType tma_dtype(int dt) {
  return dt == GE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                      : (dt == GE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

// 3-D tensor (d0 contiguous, d1, d2) with a (b0, b1, 1) box
bool encode3d(CUtensorMap *m, int dt, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2,
              uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = static_cast<uint64_t>(esize(dt));
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, tma_dtype(dt), 3, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// EW-column boxes: 16-bit rows are 64 bytes, fp32 rows 128 bytes
CUtensorMapSwizzle epi_swizzle(int dt) {
  return dt == GE_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------ configuration --
struct Layout {
  int cg = 0, bn = 0, stages = 0, aux_stages = 0, grid = 0, num_tiles = 0;
  int warps = 4;      // epilogue warps (4 or 8)
  const void *fn = nullptr;  // the kernel (chosen by configure)
  int smem = 0;       // dynamic smem requested at launch
  int smem_used = 0;  // bytes the layout occupies
  int num_m_blk = 0, num_n_blk = 0, num_kb = 0, raster_group = 0;
  int num_full = 0;   // tiles launched full width (the rest: halves of split tiles)
  uint32_t off_A = 0, off_B = 0, off_aux = 0, off_out = 0, off_bar = 0;
  uint32_t aux_stage_bytes = 0, out_stage_bytes = 0;
  uint32_t aux_off[GE_MAX_TMA_AUX] = {}, out_off[GE_MAX_OUT] = {};
  uint32_t tx_bytes = 0, aux_tx_bytes = 0;
};

constexpr int kBarBlock = 1024;
constexpr int kAlignSlack = 1024;

// Shared-memory layout for (cg, bn) and a program; stages = 0 picks the most
// that fit.  Epilogue staging is per group of 4 epilogue warps: aux slots
// (one kEpiRows x EW box per aux tensor) and output boxes (one per output).
// The aux prefetch gets the deepest ring (up to max_aux slots per group) that
// still leaves min_main mainloop stages.  Returns GE_ERR_SMEM if fewer than 2
// (or the requested count) fit.
int make_layout(Layout *Lo, int cg, int bn, int want_stages, const EpiProgram &P, int max_smem,
                int max_aux = 4, int min_main = 5, int warps = 4) {
  const uint32_t a_bytes = BM * BK * 2;
  const uint32_t b_bytes = static_cast<uint32_t>(bn / cg) * BK * 2;
  uint32_t aux_stage = 0, out_stage = 0;
  for (int t = 0; t < P.n_tma_aux; ++t) {
    Lo->aux_off[t] = aux_stage;
    aux_stage += uint32_t(kEpiRows) * EW * esize(P.tma_aux_dtype[t]);
  }
  for (int o = 0; o < P.n_out; ++o) {
    Lo->out_off[o] = out_stage;
    out_stage += uint32_t(kEpiRows) * EW * esize(P.out_dtype[o]);
  }
  const int groups = warps / 4;
  auto stages_with = [&](int sa) {
    const int64_t epi = int64_t(groups) * sa * aux_stage + int64_t(groups) * out_bufs_for(warps) * out_stage;
    const int64_t room = int64_t(max_smem) - kAlignSlack - kBarBlock - epi;
    const int s = room > 0 ? static_cast<int>(room / (a_bytes + b_bytes)) : 0;
    return std::min(s, kMaxStages);
  };
  // 4 warps: at least 2 aux stages; 8 warps (each warp's steps twice as far
  // apart in time) may go down to 1
  const int min_sa = warps == 8 ? 1 : 2;
  // a requested stage count takes the place of min_main: the aux ring is the
  // deepest that still leaves room for it
  const int need_main = want_stages > 0 ? want_stages : min_main;
  int sa = 1, stages = stages_with(1);
  if (P.n_tma_aux > 0) {
    sa = min_sa;
    stages = stages_with(min_sa);
    for (int cand = std::min(max_aux, kMaxAuxStages); cand > min_sa; --cand)
      if (stages_with(cand) >= need_main) {
        sa = cand;
        stages = stages_with(cand);
        break;
      }
  }
  if (want_stages > 0) {
    if (want_stages > stages || want_stages > kMaxStages) return GE_ERR_SMEM;
    stages = want_stages;
  }
  if (stages < 2) return GE_ERR_SMEM;
  Lo->cg = cg;
  Lo->bn = bn;
  Lo->stages = stages;
  Lo->aux_stages = sa;
  Lo->aux_stage_bytes = aux_stage;
  Lo->out_stage_bytes = out_stage;
  Lo->off_A = 0;
  Lo->off_B = stages * a_bytes;
  Lo->off_aux = Lo->off_B + stages * b_bytes;
  Lo->off_out = Lo->off_aux + groups * sa * aux_stage;
  Lo->off_bar = Lo->off_out + groups * out_bufs_for(warps) * out_stage;
  Lo->warps = warps;
  Lo->smem_used = static_cast<int>(Lo->off_bar + kBarBlock + kAlignSlack);
  // Always request the whole opt-in shared memory: exactly one CTA per SM, so
  // co-resident CTAs never compete for TMEM columns (a CTA blocked in
  // tcgen05.alloc behind another cluster's CTA could otherwise deadlock).
  Lo->smem = max_smem;
  Lo->tx_bytes = static_cast<uint32_t>(cg) * (a_bytes + b_bytes);
  Lo->aux_tx_bytes = aux_stage;
  return GE_OK;
}

}  // namespace

// ------------------------------------------------------------------- plan --
constexpr int kGroupSlots = 4;  // problem tables of a grouped plan, used in turn

struct gemm_epi_plan {
  int64_t L = 0, M = 0, N = 0, K = 0;
  ge_dtypes dt{};
  ge_dag dag{};
  ge_options opt{};
  int a_mn = 0, b_k = 0, cd_m = 0;  // operand / epilogue majors (from the options)
  int device = 0, num_sms = 0, max_smem = 0;
  uint32_t *status = nullptr;
  EpiProgram prog{}, prog_acc{};
  int epi = -1, epi_acc = -1;  // catalog entries (-1, -2: interpreter; -3: compiled at plan time)
  int interp_epi = -1;          // the interpreter variant for this program (-1 or -2)
  Layout lay, lay_acc;
  KParams kp{}, kp_acc{};
  // pointers the cached tensor maps were encoded for
  const void *mA = nullptr, *mB = nullptr;
  const void *mAux[GE_MAX_TMA_AUX] = {};
  void *mOut[GE_MAX_OUT] = {};
  bool maps_ok = false;
  const void *aA = nullptr, *aB = nullptr;
  void *aWs = nullptr;
  bool acc_maps_ok = false;
  // grouped GEMM (n_groups > 0)
  int n_groups = 0;
  std::vector<ge_problem> problems;
  std::vector<int> order;           // problem of each table entry (most k-blocks first)
  GroupDesc *d_desc = nullptr;      // kGroupSlots tables of n_groups entries, device
  GroupDesc *h_desc = nullptr;      // their pinned host staging
  int4 *d_tiles = nullptr;          // per tile {table entry, m block, n block, k blocks}
  cudaEvent_t ev[kGroupSlots] = {};  // recorded after the latest run that read each table
  bool ev_used[kGroupSlots] = {};
  cudaStream_t ev_stream[kGroupSlots] = {};  // the stream of that run
  int slot = -1;                    // table of the latest run
  std::vector<const void *> slot_ptrs[kGroupSlots];  // pointers each table was built for

  ~gemm_epi_plan() {
    for (int s = 0; s < kGroupSlots; ++s)
      if (ev[s]) {
        if (ev_used[s]) cudaEventSynchronize(ev[s]);
        cudaEventDestroy(ev[s]);
      }
    if (d_desc) cudaFree(d_desc);
    if (d_tiles) cudaFree(d_tiles);
    if (h_desc) cudaFreeHost(h_desc);
    cudaGetLastError();
  }
};

namespace {

// epi code of a kernel compiled at plan time for the plan's own program
constexpr int kEpiSpecialized = -3;
// internal status: the runtime compiler failed (the plan falls back to the
// interpreter); never returned through the ABI
constexpr int GE_ERR_JIT = -100;

const void *gemm_kernel(int cg, int bn, int epi, int warps) {
  if (cg == 1 && bn == 64) return gemm_kernel_cg1_n64(epi, warps);
  if (cg == 1 && bn == 128) return gemm_kernel_cg1_n128(epi, warps);
  if (cg == 1 && bn == 256) return gemm_kernel_cg1_n256(epi, warps);
  if (cg == 2 && bn == 128) return gemm_kernel_cg2_n128(epi, warps);
  if (cg == 2 && bn == 256) return gemm_kernel_cg2_n256(epi, warps);
  return nullptr;
}

const void *resolve_kernel(gemm_epi_plan *pl, int cg, int bn, int epi, int warps,
                           const EpiProgram *P) {
  (void)pl;
  if (epi != kEpiSpecialized) return gemm_kernel(cg, bn, epi, warps);
  std::string log;
  const void *fn = jit_gemm_kernel(*P, cg, bn, warps, &log);
  if (!fn && log_enabled())
    std::fprintf(stderr, "[gemm_epi] run-time compilation failed, using the interpreter: %s\n",
                 log.c_str());
  return fn;
}

// `attr` has room for two attributes: the cluster shape and, with `pdl`,
// programmatic stream serialization (the kernel may start while the
// previous kernel on the stream finishes; it waits in griddepcontrol.wait
// before touching global memory).
cudaLaunchConfig_t launch_config(const Layout &Lo, cudaStream_t s, cudaLaunchAttribute *attr,
                                 bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(Lo.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads_for(Lo.warps)));
  cfg.dynamicSmemBytes = static_cast<size_t>(Lo.smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (Lo.cg > 1) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(Lo.cg);
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    ++cfg.numAttrs;
  }
  if (pdl) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  if (cfg.numAttrs == 0) cfg.attrs = nullptr;
  return cfg;
}

cudaError_t launch_gemm(const Layout &Lo, int epi, const KParams &kp, cudaStream_t s, bool pdl) {
  (void)epi;
  const void *fn = Lo.fn;
  if (!fn) return cudaErrorInvalidDeviceFunction;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(Lo, s, attr, pdl);
  void *args[] = {const_cast<KParams *>(&kp)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Whether the last wave of `tiles` full tiles on `units` CTAs (pairs) is split
// into half-width tiles: when it would leave at least half of them idle, its
// r tiles become 2r halves (one per CTA at most), so the wave takes about
// half as long.  Needs whole 32-column epilogue steps per warp in a half
// (BN >= 128) and whole 64-column B atoms per CTA in a half (BN / cg >= 128,
// or K-major B, which loads whole boxes).
bool split_tail(int64_t tiles, int64_t units, int cg, int bn, bool b_k) {
  const int64_t r = tiles % units;
  return r > 0 && 2 * r <= units && bn >= 128 && (b_k || bn / cg >= 128);
}

// Rough cost model in SM clocks: waves x per-tile mainloop, where a k-block
// costs the larger of its tensor-core time (2*BN clocks for 128 x BN x 64 at
// 8192 flop/clk/SM, the rate the pipe sustains when fed back to back) and
// its operand fill time at
// ~48 B/clk/SM of L2 bandwidth when every SM is busy (measured: per-SM
// throughput drops by a third from 38 to 152 active SMs with 32 KiB per
// k-block).
double est_kblock_cycles(int cg, int bn) {
  const double mma = 2.0 * bn;
  const double fill = double((BM + bn / cg) * BK * 2) / 48.0;
  return std::max(mma, fill);
}

double est_cycles(const gemm_epi_plan *pl, int cg, int bn, int units) {
  const int64_t mt = (pl->M + BM * cg - 1) / (BM * cg);
  const int64_t nt = (pl->N + bn - 1) / bn;
  const int64_t tiles = pl->L * mt * nt;
  const int64_t kb = (pl->K + BK - 1) / BK;
  const double per_tile = kb * est_kblock_cycles(cg, bn);
  const bool split = (pl->opt.debug_flags & GE_DEBUG_NO_TAIL_SPLIT) == 0u &&
                     split_tail(tiles, units, cg, bn, pl->b_k != 0);
  const double waves = split ? double(tiles / units) + 0.5 : double((tiles + units - 1) / units);
  return waves * per_tile + (bn / CH) * 300.0;
}

// Epilogue warps: the option, else 8 — two warps per lane quarter overlap
// each other's waits: with built-in epilogues measured equal or faster on
// every workload (up to 1.5x where the epilogue outweighs a short mainloop;
// at 8192^3, where the epilogue hides under a 128-k-block mainloop, 620.5-
// 620.6 against 622.9-626.6 us over 20 launches and 683-691 against 691-696
// over 300, four interleaved repetitions each); with the interpreter, which
// then spills a few registers, 1.13x to 1.27x faster on transcendental and
// multi-output epilogues and 4 % slower on a cheap one.  The interpreter of
// programs with more than four live values holds twice the registers and
// runs on 4.
int pick_epi_warps(const gemm_epi_plan *pl, int *warps) {
  const int w = pl->opt.epi_warps;
  if (w != 0 && w != 4 && w != 8) return GE_ERR_INVALID;
  if (w == 8 && pl->epi == -2) return GE_ERR_UNSUPPORTED;
  *warps = w ? w : (pl->epi == -2 ? 4 : 8);
  return GE_OK;
}

int configure(gemm_epi_plan *pl) {
  const ge_options &o = pl->opt;
  if (o.cta_group != 0 && o.cta_group != 1 && o.cta_group != 2) return GE_ERR_INVALID;
  if (o.tile_n != 0 && o.tile_n != 64 && o.tile_n != 128 && o.tile_n != 256) return GE_ERR_INVALID;
  if (o.stages < 0 || o.stages > kMaxStages || o.max_ctas < 0 || o.raster_group < 0 ||
      o.timeout_ms < 0)
    return GE_ERR_INVALID;
  const int cand[5][2] = {{2, 256}, {2, 128}, {1, 256}, {1, 128}, {1, 64}};
  int best = -1;
  double best_c = 0;
  for (int c = 0; c < 5; ++c) {
    const int cg = cand[c][0], bn = cand[c][1];
    if (o.cta_group && o.cta_group != cg) continue;
    if (o.tile_n && o.tile_n != bn) continue;
    int sms = pl->num_sms;
    if (o.max_ctas) sms = std::min(sms, o.max_ctas);
    if (sms < cg) continue;
    const int units = sms / cg;
    const double cost = est_cycles(pl, cg, bn, units);
    if (best < 0 || cost < best_c * 0.98) {
      best = c;
      best_c = cost;
    }
  }
  if (best < 0) return GE_ERR_INVALID;  // e.g. cta_group 2 with tile_n 64
  const int cg = cand[best][0], bn = cand[best][1];

  int warps = 0;
  int st = pick_epi_warps(pl, &warps);
  if (st != GE_OK) return st;
  st = make_layout(&pl->lay, cg, bn, o.stages, pl->prog, pl->max_smem, 4, 5, warps);
  if (st != GE_OK) return st;
  // the unfused path's GEMM stores fp32 accum: a built-in epilogue on 8 warps
  st = make_layout(&pl->lay_acc, cg, bn, o.stages, pl->prog_acc, pl->max_smem, 4, 5,
                   pl->epi_acc >= 0 ? 8 : 4);
  if (st != GE_OK) return st;

  for (Layout *Lo : {&pl->lay, &pl->lay_acc}) {
    Lo->num_m_blk = static_cast<int>((pl->M + BM * cg - 1) / (BM * cg));
    Lo->num_n_blk = static_cast<int>((pl->N + bn - 1) / bn);
    Lo->num_kb = static_cast<int>((pl->K + BK - 1) / BK);
    const int64_t tiles = pl->L * Lo->num_m_blk * int64_t(Lo->num_n_blk);
    if (tiles > (int64_t(1) << 30)) return GE_ERR_SHAPE;
    Lo->num_tiles = static_cast<int>(tiles);
    // Raster groups: all M tiles in one group when there are at most 16,
    // else 12 M tiles per group.  At 8192^3 (32 M tiles) 12 is as fast as 16
    // (647.6 against 648.1 us over 20 launches, 702.7 against 703.6 over
    // 200, four interleaved repetitions each) and 8 (652.1, 708.9) and reads
    // 6.5 % less from DRAM than 16 (1.19 against 1.27 GB per launch); with 16
    // M tiles per batch (L=8, 4096 x 4096 x 2048) one group of 16 reads 6 %
    // less than 12 + 4 (0.62 against 0.66 GB) and runs 0.3 % faster.
    Lo->raster_group = o.raster_group ? o.raster_group : (Lo->num_m_blk <= 16 ? 16 : 12);
    int sms = pl->num_sms;
    if (o.max_ctas) sms = std::min(sms, o.max_ctas);
    int units = std::max(1, sms / cg);
    const void *fn = resolve_kernel(pl, cg, bn, Lo == &pl->lay ? pl->epi : pl->epi_acc,
                                    Lo->warps, Lo == &pl->lay ? &pl->prog : &pl->prog_acc);
    if (!fn) return pl->epi == kEpiSpecialized && Lo == &pl->lay ? GE_ERR_JIT : GE_ERR_INVALID;
    Lo->fn = fn;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Lo->smem) != cudaSuccess)
      return GE_ERR_CUDA;
    if (cg > 1) {
      int clusters = 0;
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = launch_config(*Lo, nullptr, attr);
      cfg.gridDim = dim3(static_cast<unsigned>(cg));
      if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess && clusters > 0)
        units = std::min(units, clusters);
      cudaGetLastError();
    }
    Lo->num_full = Lo->num_tiles;
    if ((o.debug_flags & GE_DEBUG_NO_TAIL_SPLIT) == 0u &&
        split_tail(tiles, units, cg, bn, pl->b_k != 0)) {
      const int64_t r = tiles % units;
      Lo->num_full = static_cast<int>(tiles - r);
      Lo->num_tiles = static_cast<int>(tiles + r);
    }
    units = static_cast<int>(std::min<int64_t>(units, Lo->num_tiles));
    Lo->grid = units * cg;
  }
  return GE_OK;
}

void fill_params(const gemm_epi_plan *pl, const Layout &Lo, const EpiProgram &P, KParams *kp) {
  std::memset(static_cast<void *>(kp), 0, sizeof(*kp));
  kp->status = pl->status;
  kp->prog = P;
  kp->L = static_cast<int32_t>(pl->L);
  kp->M = static_cast<int32_t>(pl->M);
  kp->N = static_cast<int32_t>(pl->N);
  kp->K = static_cast<int32_t>(pl->K);
  kp->ab_bf16 = pl->dt.ab == GE_BF16;
  kp->num_m_blk = Lo.num_m_blk;
  kp->num_n_blk = Lo.num_n_blk;
  kp->num_tiles = Lo.num_tiles;
  kp->num_full = Lo.num_full;
  kp->num_kb = Lo.num_kb;
  kp->raster_group = Lo.raster_group;
  kp->stages = Lo.stages;
  kp->aux_stages = Lo.aux_stages;
  kp->off_A = Lo.off_A;
  kp->off_B = Lo.off_B;
  kp->off_aux = Lo.off_aux;
  kp->off_out = Lo.off_out;
  kp->off_bar = Lo.off_bar;
  kp->aux_stage_bytes = Lo.aux_stage_bytes;
  kp->out_stage_bytes = Lo.out_stage_bytes;
  for (int i = 0; i < GE_MAX_TMA_AUX; ++i) kp->aux_off[i] = Lo.aux_off[i];
  for (int i = 0; i < GE_MAX_OUT; ++i) kp->out_off[i] = Lo.out_off[i];
  kp->tx_bytes = Lo.tx_bytes;
  // a half tile: half the B bytes per CTA (N-major B), or the same whole
  // boxes (K-major B)
  const uint32_t b_bytes = static_cast<uint32_t>(Lo.bn / std::max(Lo.cg, 1)) * BK * 2;
  kp->tx_bytes_half = pl->b_k ? Lo.tx_bytes : Lo.tx_bytes - static_cast<uint32_t>(Lo.cg) * (b_bytes / 2);
  kp->aux_tx_bytes = Lo.aux_tx_bytes;
  // B tile in shared memory: 64-column (128-byte) swizzle atoms of 64 k-rows
  // (8 KiB apart), 8-row groups 1 KiB apart
  kp->b_lbo = 8192;
  kp->b_sbo = 1024;
  const int tmo = pl->opt.timeout_ms ? pl->opt.timeout_ms : 1000;
  kp->timeout_ns = static_cast<uint64_t>(tmo) * 1000000ull;
  kp->debug_flags = pl->opt.debug_flags;
  kp->a_mn = pl->a_mn;
  kp->b_k = pl->b_k;
  kp->cd_m = pl->cd_m;
}

// A and B tensor maps of one (L, M, N, K) problem.  K-major A: (K, M, L), box
// 64 x the rows one CTA fetches; M-major A: (M, K, L), box 64 x 64 (one of
// the tile's two 64-row atoms); N-major B: (N, K, L), box 64 x 64 (one 64-column
// atom); K-major B: (K, N, L), box 64 x the CTA's tile columns.
bool encode_ab_maps(const gemm_epi_plan *pl, CUtensorMap *tA, CUtensorMap *tB, const void *A,
                    const void *B, uint64_t L, uint64_t M, uint64_t N, uint64_t K) {
  const int ab = pl->dt.ab;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  const bool okA = pl->a_mn ? encode3d(tA, ab, A, M, K, L, 64, BK, sw, l2)
                            : encode3d(tA, ab, A, K, M, L, BK, BM, sw, l2);
  const bool okB = pl->b_k ? encode3d(tB, ab, B, K, N, L, BK,
                                      static_cast<uint32_t>(pl->lay.bn / pl->lay.cg), sw, l2)
                           : encode3d(tB, ab, B, N, K, L, 64, BK, sw, l2);
  return okA && okB;
}

bool encode_operands(const gemm_epi_plan *pl, KParams *kp, const void *A, const void *B) {
  return encode_ab_maps(pl, &kp->tmA, &kp->tmB, A, B, pl->L, pl->M, pl->N, pl->K);
}

// An epilogue tensor's map: N-major (N, M, L) with EW x kEpiRows swizzled
// boxes, or M-major (M, N, L) with kEpiRows x EW plain boxes: one box holds a
// 32-column step of all of a CTA's accumulator rows.  The unfused path's fp32
// workspace follows the epilogue tensors' order.
bool encode_epi_map(const gemm_epi_plan *pl, CUtensorMap *m, int dt, const void *ptr, uint64_t L,
                    uint64_t M, uint64_t N) {
  if (pl->cd_m)
    return encode3d(m, dt, ptr, M, N, L, kEpiRows, EW, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  return encode3d(m, dt, ptr, N, M, L, EW, kEpiRows, epi_swizzle(dt),
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

bool encode_epilogue_map(const gemm_epi_plan *pl, CUtensorMap *m, int dt, const void *ptr) {
  return encode_epi_map(pl, m, dt, ptr, pl->L, pl->M, pl->N);
}

// Operand and epilogue majors from the options (all row-major without options).
int read_majors(gemm_epi_plan *pl, const ge_options *o) {
  if (!o) return GE_OK;
  for (int v : {o->a_major, o->b_major, o->cd_major})
    if (v != GE_ROW_MAJOR && v != GE_COL_MAJOR) return GE_ERR_INVALID;
  pl->a_mn = o->a_major == GE_COL_MAJOR;
  pl->b_k = o->b_major == GE_COL_MAJOR;
  pl->cd_m = o->cd_major == GE_COL_MAJOR;
  // one CTA pair per cluster: no cluster multicast of operand tiles
  if (o->cluster_n != 0 && o->cluster_n != 1) return GE_ERR_UNSUPPORTED;
  return GE_OK;
}

// The contiguous dimension of every tensor must be whole 16-byte units.
int check_alignment(const gemm_epi_plan *pl, const ge_dtypes *dt, int64_t M, int64_t N, int64_t K) {
  const int64_t ea = esize(dt->ab);
  if (((pl->a_mn ? M : K) * ea) % 16 != 0 || ((pl->b_k ? K : N) * ea) % 16 != 0)
    return GE_ERR_MISALIGNED;
  for (int o = 0; o < dt->n_out; ++o) {
    if ((N * esize(dt->out[o])) % 16 != 0) return GE_ERR_MISALIGNED;
    if (pl->cd_m && (M * esize(dt->out[o])) % 16 != 0) return GE_ERR_MISALIGNED;
  }
  for (int s = 0; s < dt->n_aux; ++s) {
    if ((N * esize(dt->aux[s])) % 16 != 0) return GE_ERR_MISALIGNED;
    if (pl->cd_m && (M * esize(dt->aux[s])) % 16 != 0) return GE_ERR_MISALIGNED;
  }
  return GE_OK;
}

int check_device(int *dev, int *sms, int *max_smem) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_ARCH;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_ARCH;
  }
  if (major != 10 || minor != 3) return GE_ERR_ARCH;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) != cudaSuccess)
    return GE_ERR_CUDA;
  return GE_OK;
}

int check_run_args(const gemm_epi_plan *pl, const void *A, const void *B, const void *const *aux,
                   const float *scalars, void *const *outs) {
  if (!A || !B || !outs) return GE_ERR_MISSING_ARG;
  if (pl->dt.n_scalar > 0 && !scalars) return GE_ERR_MISSING_ARG;
  if (!aligned16(A) || !aligned16(B)) return GE_ERR_MISALIGNED;
  const EpiProgram &P = pl->prog;
  if ((P.n_tma_aux + P.n_bcast + P.n_cbcast) > 0 && !aux) return GE_ERR_MISSING_ARG;
  for (int t = 0; t < P.n_tma_aux; ++t) {
    const void *p = aux[P.tma_aux_slot[t]];
    if (!p) return GE_ERR_MISSING_ARG;
    if (!aligned16(p)) return GE_ERR_MISALIGNED;
  }
  for (int b = 0; b < P.n_bcast; ++b) {
    const void *p = aux[P.bcast_slot[b]];
    if (!p) return GE_ERR_MISSING_ARG;
    if (!aligned16(p)) return GE_ERR_MISALIGNED;
  }
  for (int b = 0; b < P.n_cbcast; ++b) {
    const void *p = aux[P.cbcast_slot[b]];
    if (!p) return GE_ERR_MISSING_ARG;
    if (!aligned16(p)) return GE_ERR_MISALIGNED;
  }
  for (int o = 0; o < pl->dt.n_out; ++o) {
    if (!outs[o]) return GE_ERR_MISSING_ARG;
    if (!aligned16(outs[o])) return GE_ERR_MISALIGNED;
  }
  return GE_OK;
}

void log_plan(const gemm_epi_plan *pl) {
  const Layout &Lo = pl->lay;
  std::fprintf(stderr,
               "[gemm_epi] L=%lld M=%lld N=%lld K=%lld: cta_group=%d tile=%dx%dx%d stages=%d "
               "aux_stages=%d grid=%d tiles=%d smem=%d program=%d ins/%d regs epilogue=%s\n",
               (long long)pl->L, (long long)pl->M, (long long)pl->N, (long long)pl->K, Lo.cg,
               BM * Lo.cg, Lo.bn, BK, Lo.stages, Lo.aux_stages, Lo.grid, Lo.num_tiles, Lo.smem_used,
               pl->prog.n_ins, pl->prog.n_regs,
               pl->epi >= 0                 ? catalog::kEntries[pl->epi].name
               : pl->epi == kEpiSpecialized ? "compiled for this program"
                                            : "interpreter");
}

}  // namespace

// ------------------------------------------------------------- C ABI --
extern "C" {

int gemm_epi_validate(const ge_dtypes *dtypes, const ge_dag *dag) {
  int st = validate_impl(dtypes, dag);
  if (st != GE_OK) return st;
  return compile_program(*dtypes, *dag).status;
}

int gemm_epi_plan_create_ex(gemm_epi_plan **plan, int64_t L, int64_t M, int64_t N, int64_t K,
                            const ge_dtypes *dtypes, const ge_dag *dag, const ge_options *opts) {
  if (!plan) return GE_ERR_INVALID;
  *plan = nullptr;
  int st = validate_impl(dtypes, dag);
  if (st != GE_OK) return st;
  if (L <= 0 || M <= 0 || N <= 0 || K <= 0) return GE_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1 ||
      L > (int64_t(1) << 31) - 1)
    return GE_ERR_SHAPE;
  gemm_epi_plan *pl = new (std::nothrow) gemm_epi_plan();
  if (!pl) return GE_ERR_INVALID;
  st = read_majors(pl, opts);
  if (st == GE_OK) st = check_alignment(pl, dtypes, M, N, K);
  if (st != GE_OK) {
    delete pl;
    return st;
  }
  pl->L = L;
  pl->M = M;
  pl->N = N;
  pl->K = K;
  pl->dt = *dtypes;
  pl->dag = *dag;
  if (opts) pl->opt = *opts;
  {
    const CompileResult cr = compile_program(*dtypes, *dag);
    st = cr.status;
    pl->prog = cr.prog;
  }
  if (st == GE_OK) {
    pl->prog_acc = program_store_accum();
    const bool interp = (pl->opt.debug_flags & GE_DEBUG_FORCE_INTERPRETER) != 0u;
    pl->epi = pick_executor(pl->prog, interp);
    pl->interp_epi = pl->prog.n_regs > 4 ? -2 : -1;
    pl->epi_acc = pick_executor(pl->prog_acc, interp);
    st = check_device(&pl->device, &pl->num_sms, &pl->max_smem);
    if (st == GE_OK && pl->epi < 0 && !interp && pl->opt.specialize >= 0 && jit_available())
      pl->epi = kEpiSpecialized;
  }
  if (st == GE_OK) {
    void *sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_ge_status) != cudaSuccess) st = GE_ERR_CUDA;
    pl->status = static_cast<uint32_t *>(sym);
  }
  if (st == GE_OK) st = configure(pl);
  if (st == GE_ERR_JIT) {  // the runtime compiler failed: the interpreter
    pl->epi = pl->interp_epi;
    st = configure(pl);
  }
  if (st == GE_OK && !encode_fn()) st = GE_ERR_CUDA;
  if (st != GE_OK) {
    cudaGetLastError();
    delete pl;
    return st;
  }
  fill_params(pl, pl->lay, pl->prog, &pl->kp);
  fill_params(pl, pl->lay_acc, pl->prog_acc, &pl->kp_acc);
  if (log_enabled()) log_plan(pl);
  *plan = pl;
  return GE_OK;
}

int gemm_epi_plan_create(gemm_epi_plan **plan, int64_t L, int64_t M, int64_t N, int64_t K,
                         const ge_dtypes *dtypes, const ge_dag *dag) {
  return gemm_epi_plan_create_ex(plan, L, M, N, K, dtypes, dag, nullptr);
}

void gemm_epi_plan_destroy(gemm_epi_plan *plan) { delete plan; }

int gemm_epi_plan_info(const gemm_epi_plan *pl, ge_plan_info *info) {
  if (!pl || !info) return GE_ERR_INVALID;
  info->cta_group = pl->lay.cg;
  info->tile_m = BM * pl->lay.cg;
  info->tile_n = pl->lay.bn;
  info->tile_k = BK;
  info->stages = pl->lay.stages;
  info->epi_chunk = CH;
  info->aux_stages = pl->lay.aux_stages;
  info->grid = pl->lay.grid;
  info->num_tiles = pl->lay.num_tiles;
  info->smem_bytes = pl->lay.smem_used;
  info->n_instr = pl->prog.n_ins;
  info->n_regs = pl->prog.n_regs;
  info->num_sms = pl->num_sms;
  info->epi_variant = pl->epi;
  info->cluster_n = 1;
  info->epi_warps = pl->lay.warps;
  // the group size in effect: a batched launch with fewer M tiles than the
  // group size runs them all as one group
  info->raster_group = pl->n_groups ? pl->lay.raster_group
                                    : std::min(pl->lay.raster_group, pl->lay.num_m_blk);
  return GE_OK;
}

int gemm_epi_run(gemm_epi_plan *pl, const void *A, const void *B, const void *const *aux,
                 const float *scalars, void *const *outs, void *stream) {
  if (!pl || pl->n_groups) return GE_ERR_INVALID;
  int st = check_run_args(pl, A, B, aux, scalars, outs);
  if (st != GE_OK) return st;
  KParams &kp = pl->kp;
  const EpiProgram &P = pl->prog;
  // re-encode tensor maps only when a pointer changed
  bool same = pl->maps_ok && pl->mA == A && pl->mB == B;
  for (int t = 0; same && t < P.n_tma_aux; ++t) same = pl->mAux[t] == aux[P.tma_aux_slot[t]];
  for (int o = 0; same && o < pl->dt.n_out; ++o) same = pl->mOut[o] == outs[o];
  if (!same) {
    pl->maps_ok = false;
    if (!encode_operands(pl, &kp, A, B)) return GE_ERR_CUDA;
    for (int t = 0; t < P.n_tma_aux; ++t)
      if (!encode_epilogue_map(pl, &kp.tmAux[t], P.tma_aux_dtype[t], aux[P.tma_aux_slot[t]]))
        return GE_ERR_CUDA;
    for (int o = 0; o < pl->dt.n_out; ++o)
      if (!encode_epilogue_map(pl, &kp.tmOut[o], P.out_dtype[o], outs[o])) return GE_ERR_CUDA;
    pl->mA = A;
    pl->mB = B;
    for (int t = 0; t < P.n_tma_aux; ++t) pl->mAux[t] = aux[P.tma_aux_slot[t]];
    for (int o = 0; o < pl->dt.n_out; ++o) pl->mOut[o] = outs[o];
    pl->maps_ok = true;
  }
  for (int b = 0; b < P.n_bcast; ++b) kp.bcast_ptr[b] = aux[P.bcast_slot[b]];
  for (int b = 0; b < P.n_cbcast; ++b) kp.cbcast_ptr[b] = aux[P.cbcast_slot[b]];
  for (int s = 0; s < pl->dt.n_scalar; ++s) kp.prog.scalars[s] = scalars[s];
  const cudaError_t e = launch_gemm(pl->lay, pl->epi, kp, static_cast<cudaStream_t>(stream),
                                    pl->opt.no_pdl == 0);
  return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

size_t gemm_epi_unfused_workspace_bytes(const gemm_epi_plan *pl) {
  if (!pl || pl->n_groups) return 0;
  return static_cast<size_t>(pl->L) * static_cast<size_t>(pl->M) * static_cast<size_t>(pl->N) * 4u;
}

int gemm_epi_run_unfused(gemm_epi_plan *pl, const void *A, const void *B, const void *const *aux,
                         const float *scalars, void *const *outs, void *workspace,
                         size_t workspace_bytes, void *stream) {
  if (!pl || pl->n_groups) return GE_ERR_INVALID;
  int st = check_run_args(pl, A, B, aux, scalars, outs);
  if (st != GE_OK) return st;
  if (!workspace || !aligned16(workspace) || workspace_bytes < gemm_epi_unfused_workspace_bytes(pl))
    return GE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // launch 1: GEMM, accumulator stored as fp32
  KParams &ka = pl->kp_acc;
  if (!(pl->acc_maps_ok && pl->aA == A && pl->aB == B && pl->aWs == workspace)) {
    pl->acc_maps_ok = false;
    if (!encode_operands(pl, &ka, A, B)) return GE_ERR_CUDA;
    if (!encode_epilogue_map(pl, &ka.tmOut[0], GE_F32, workspace)) return GE_ERR_CUDA;
    pl->aA = A;
    pl->aB = B;
    pl->aWs = workspace;
    pl->acc_maps_ok = true;
  }
  cudaError_t e = launch_gemm(pl->lay_acc, pl->epi_acc, ka, s, pl->opt.no_pdl == 0);
  if (e != cudaSuccess) return GE_ERR_CUDA;
  // launch 2: the epilogue program, elementwise
  EwParams ep;
  std::memset(static_cast<void *>(&ep), 0, sizeof(ep));
  const EpiProgram &P = pl->prog;
  ep.acc = static_cast<const float *>(workspace);
  for (int t = 0; t < P.n_tma_aux; ++t) ep.aux_ptr[t] = aux[P.tma_aux_slot[t]];
  for (int b = 0; b < P.n_bcast; ++b) ep.bcast_ptr[b] = aux[P.bcast_slot[b]];
  for (int b = 0; b < P.n_cbcast; ++b) ep.cbcast_ptr[b] = aux[P.cbcast_slot[b]];
  ep.M = static_cast<int32_t>(pl->M);
  for (int o = 0; o < pl->dt.n_out; ++o) ep.out_ptr[o] = outs[o];
  ep.prog = P;
  for (int i = 0; i < pl->dt.n_scalar; ++i) ep.prog.scalars[i] = scalars[i];
  ep.N = static_cast<int32_t>(pl->N);
  ep.cd_m = pl->cd_m;
  // units of 8 elements along the contiguous dimension: 8 columns of one of
  // the L*M rows, or (M-major) 8 rows of one of the L*N columns
  ep.rows = pl->cd_m ? pl->L * pl->N : pl->L * pl->M;
  ep.chunks_per_row = static_cast<int32_t>(((pl->cd_m ? pl->M : pl->N) + kEwCols - 1) / kEwCols);
  const int64_t units = ep.rows * ep.chunks_per_row;
  const int64_t blocks = (units + kEwThreads - 1) / kEwThreads;
  const int grid = static_cast<int>(std::min<int64_t>(blocks, int64_t(pl->num_sms) * 16));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max(grid, 1)));
  cfg.blockDim = dim3(kEwThreads);
  cfg.stream = s;
  void *args[] = {&ep};
  e = cudaLaunchKernelExC(&cfg, ew_kernel(pl->epi == kEpiSpecialized ? pl->interp_epi : pl->epi),
                         args);
  return e == cudaSuccess ? GE_OK : GE_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------ grouped GEMM --
namespace {

// Cost of one tile of a grouped problem in SM clocks: the mainloop (the
// model of est_cycles) or the epilogue, whichever is slower, since the two
// overlap across consecutive tiles, plus a fixed cost per tile.  The epilogue
// and fixed terms are fitted to measured launches of many short problems,
// whose tiles are short: 3000 clocks per 16-column chunk with 4 epilogue
// warps (half that with 8), 4000 per tile.  (Measured: the grouped
// notebook's 50 problems run in 32.2 us on 128 x 128 single-CTA tiles
// against 37.1 on 256 x 256 pair tiles; 12 ragged problems 18.6 against
// 20.0 on 256 x 128 pairs.)
double grouped_tile_cycles(int64_t K, int cg, int bn, int warps) {
  const int64_t kb = (K + BK - 1) / BK;
  const double fill = double((BM + bn / cg) * BK * 2) / 48.0;
  const double main = kb * std::max(2.0 * bn, fill);
  return std::max(main, (bn / CH) * 3000.0 * 4.0 / warps) + 4000.0;
}

// The launch deals the tiles (problems with the most k-blocks first) round
// robin to the units; it lasts about as long as the busiest unit.
double est_cycles_grouped(const gemm_epi_plan *pl, const std::vector<int> &order, int cg, int bn,
                          int units, int warps) {
  std::vector<double> busy(static_cast<size_t>(units), 0.0);
  int64_t t = 0;
  for (int g : order) {
    const ge_problem &pr = pl->problems[g];
    const int64_t tiles = ((pr.M + BM * cg - 1) / (BM * cg)) * ((pr.N + bn - 1) / bn);
    const double c = grouped_tile_cycles(pr.K, cg, bn, warps);
    // whole rounds of the deal add c to every unit; the rest to the next ones
    const int64_t rounds = tiles / units, rest = tiles % units;
    for (int u = 0; u < units; ++u) busy[u] += rounds * c;
    for (int64_t r = 0; r < rest; ++r) busy[(t + r) % units] += c;
    t = (t + tiles) % units;
  }
  return *std::max_element(busy.begin(), busy.end());
}

int configure_grouped(gemm_epi_plan *pl) {
  const ge_options &o = pl->opt;
  if (o.cta_group != 0 && o.cta_group != 1 && o.cta_group != 2) return GE_ERR_INVALID;
  if (o.tile_n != 0 && o.tile_n != 64 && o.tile_n != 128 && o.tile_n != 256) return GE_ERR_INVALID;
  if (o.stages < 0 || o.stages > kMaxStages || o.max_ctas < 0 || o.raster_group < 0 ||
      o.timeout_ms < 0)
    return GE_ERR_INVALID;
  const int cand[5][2] = {{2, 256}, {2, 128}, {1, 256}, {1, 128}, {1, 64}};
  int sms = pl->num_sms;
  if (o.max_ctas) sms = std::min(sms, o.max_ctas);
  // table order: problems with the most k-blocks first, so the round-robin
  // deal hands every unit its long tiles early and the short ones last
  const int n = pl->n_groups;
  pl->order.resize(n);
  for (int g = 0; g < n; ++g) pl->order[g] = g;
  std::stable_sort(pl->order.begin(), pl->order.end(), [&](int a, int b) {
    return pl->problems[a].K > pl->problems[b].K;
  });
  int warps = 0;
  int st = pick_epi_warps(pl, &warps);
  if (st != GE_OK) return st;
  int best = -1;
  double best_c = 0;
  for (int c = 0; c < 5; ++c) {
    const int cg = cand[c][0], bn = cand[c][1];
    if (o.cta_group && o.cta_group != cg) continue;
    if (o.tile_n && o.tile_n != bn) continue;
    if (sms < cg) continue;
    const double cost = est_cycles_grouped(pl, pl->order, cg, bn, sms / cg, warps);
    if (best < 0 || cost < best_c * 0.98) {
      best = c;
      best_c = cost;
    }
  }
  if (best < 0) return GE_ERR_INVALID;
  const int cg = cand[best][0], bn = cand[best][1];
  // short problems make short tiles, whose epilogue would wait on aux loads
  // issued only a few steps ahead: prefetch up to two tiles' steps of aux
  // data, keeping 4 mainloop stages
  st = make_layout(&pl->lay, cg, bn, o.stages, pl->prog, pl->max_smem,
                   std::min(kMaxAuxStages, 2 * bn / EW), 4, warps);
  if (st != GE_OK) return st;
  Layout &Lo = pl->lay;
  Lo.raster_group = o.raster_group ? o.raster_group : 8;
  int64_t tiles = 0;
  for (int j = 0; j < n; ++j) {
    const ge_problem &pr = pl->problems[pl->order[j]];
    tiles += ((pr.M + BM * cg - 1) / (BM * cg)) * ((pr.N + bn - 1) / bn);
  }
  if (tiles > (int64_t(1) << 24)) return GE_ERR_SHAPE;  // the tile table: 16 bytes a tile
  Lo.num_tiles = static_cast<int>(tiles);
  Lo.num_full = Lo.num_tiles;  // grouped tiles are never split
  const void *fn = resolve_kernel(pl, cg, bn, pl->epi, Lo.warps, &pl->prog);
  if (!fn) return pl->epi == kEpiSpecialized ? GE_ERR_JIT : GE_ERR_INVALID;
  Lo.fn = fn;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Lo.smem) != cudaSuccess)
    return GE_ERR_CUDA;
  int units = std::max(1, sms / cg);
  if (cg > 1) {
    int clusters = 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config(Lo, nullptr, attr);
    cfg.gridDim = dim3(static_cast<unsigned>(cg));
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess && clusters > 0)
      units = std::min(units, clusters);
    cudaGetLastError();
  }
  units = static_cast<int>(std::min<int64_t>(units, tiles));
  Lo.grid = units * cg;
  return GE_OK;
}

// Host copy of tile_coords: the order of one problem's tiles.
void raster_coords(int num_m_blk, int num_n_blk, int G, int r, int *mb, int *nb) {
  const int group = r / (G * num_n_blk);
  const int first_m = group * G;
  const int gsize = std::min(num_m_blk - first_m, G);
  const int rr = r - group * G * num_n_blk;
  *mb = first_m + rr % gsize;
  *nb = rr / gsize;
}

// The launch's tile sequence: every table entry's tiles in turn.
std::vector<int4> grouped_tile_table(const gemm_epi_plan *pl) {
  std::vector<int4> t;
  t.reserve(static_cast<size_t>(pl->lay.num_tiles));
  const GroupDesc *d = pl->h_desc;  // table 0 (the shapes are the same in all)
  for (int j = 0; j < pl->n_groups; ++j)
    for (int r = 0; r < d[j].tile_end - d[j].tile_begin; ++r) {
      int mb = 0, nb = 0;
      raster_coords(d[j].num_m_blk, d[j].num_n_blk, pl->lay.raster_group, r, &mb, &nb);
      t.push_back(make_int4(j, mb, nb, d[j].num_kb));
    }
  return t;
}

// The sizes and tile ranges of every table entry (the same in all tables).
void fill_group_shapes(gemm_epi_plan *pl) {
  const int n = pl->n_groups, cg = pl->lay.cg, bn = pl->lay.bn;
  for (int s = 0; s < kGroupSlots; ++s) {
    int begin = 0;
    for (int j = 0; j < n; ++j) {
      const ge_problem &pr = pl->problems[pl->order[j]];
      GroupDesc &d = pl->h_desc[s * n + j];
      std::memset(static_cast<void *>(&d), 0, sizeof(d));
      d.M = static_cast<int32_t>(pr.M);
      d.N = static_cast<int32_t>(pr.N);
      d.num_m_blk = static_cast<int32_t>((pr.M + BM * cg - 1) / (BM * cg));
      d.num_n_blk = static_cast<int32_t>((pr.N + bn - 1) / bn);
      d.num_kb = static_cast<int32_t>((pr.K + BK - 1) / BK);
      d.tile_begin = begin;
      begin += d.num_m_blk * d.num_n_blk;
      d.tile_end = begin;
      d.problem = pl->order[j];
    }
  }
}

// Encode the tensor maps and vector pointers of table `s` for one run.
bool build_group_table(gemm_epi_plan *pl, int s, const void *const *A, const void *const *B,
                       const void *const *aux, void *const *outs) {
  const EpiProgram &P = pl->prog;
  const int n = pl->n_groups, na = pl->dt.n_aux, no = pl->dt.n_out;
  for (int j = 0; j < n; ++j) {
    const int g = pl->order[j];
    const ge_problem &pr = pl->problems[g];
    GroupDesc &d = pl->h_desc[s * n + j];
    const uint64_t M = pr.M, N = pr.N, K = pr.K;
    if (!encode_ab_maps(pl, &d.tmA, &d.tmB, A[g], B[g], 1, M, N, K)) return false;
    for (int t = 0; t < P.n_tma_aux; ++t)
      if (!encode_epi_map(pl, &d.tmAux[t], P.tma_aux_dtype[t], aux[g * na + P.tma_aux_slot[t]], 1,
                          M, N))
        return false;
    for (int o = 0; o < no; ++o)
      if (!encode_epi_map(pl, &d.tmOut[o], P.out_dtype[o], outs[g * no + o], 1, M, N))
        return false;
    for (int b = 0; b < P.n_bcast; ++b) d.bcast_ptr[b] = aux[g * na + P.bcast_slot[b]];
    for (int b = 0; b < P.n_cbcast; ++b) d.cbcast_ptr[b] = aux[g * na + P.cbcast_slot[b]];
  }
  return true;
}

int check_grouped_args(const gemm_epi_plan *pl, const void *const *A, const void *const *B,
                       const void *const *aux, const float *scalars, void *const *outs) {
  if (!A || !B || !outs) return GE_ERR_MISSING_ARG;
  if (pl->dt.n_scalar > 0 && !scalars) return GE_ERR_MISSING_ARG;
  const EpiProgram &P = pl->prog;
  const int na = pl->dt.n_aux, no = pl->dt.n_out;
  if ((P.n_tma_aux + P.n_bcast + P.n_cbcast) > 0 && !aux) return GE_ERR_MISSING_ARG;
  auto check = [](const void *p) {
    return !p ? GE_ERR_MISSING_ARG : (aligned16(p) ? GE_OK : GE_ERR_MISALIGNED);
  };
  for (int g = 0; g < pl->n_groups; ++g) {
    int st = GE_OK;
    if ((st = check(A[g])) != GE_OK || (st = check(B[g])) != GE_OK) return st;
    for (int t = 0; t < P.n_tma_aux; ++t)
      if ((st = check(aux[g * na + P.tma_aux_slot[t]])) != GE_OK) return st;
    for (int b = 0; b < P.n_bcast; ++b)
      if ((st = check(aux[g * na + P.bcast_slot[b]])) != GE_OK) return st;
    for (int b = 0; b < P.n_cbcast; ++b)
      if ((st = check(aux[g * na + P.cbcast_slot[b]])) != GE_OK) return st;
    for (int o = 0; o < no; ++o)
      if ((st = check(outs[g * no + o])) != GE_OK) return st;
  }
  return GE_OK;
}

}  // namespace

extern "C" {

int gemm_epi_grouped_plan_create(gemm_epi_plan **plan, int32_t n_problems,
                                 const ge_problem *problems, const ge_dtypes *dtypes,
                                 const ge_dag *dag, const ge_options *opts) {
  if (!plan) return GE_ERR_INVALID;
  *plan = nullptr;
  int st = validate_impl(dtypes, dag);
  if (st != GE_OK) return st;
  if (!problems) return GE_ERR_INVALID;
  if (n_problems < 1 || n_problems > GE_MAX_GROUPS) return GE_ERR_SHAPE;
  for (int g = 0; g < n_problems; ++g) {
    const ge_problem &pr = problems[g];
    if (pr.M <= 0 || pr.N <= 0 || pr.K <= 0) return GE_ERR_SHAPE;
    if (pr.M > (int64_t(1) << 31) - 1 || pr.N > (int64_t(1) << 31) - 1 ||
        pr.K > (int64_t(1) << 31) - 1)
      return GE_ERR_SHAPE;
  }
  gemm_epi_plan *pl = new (std::nothrow) gemm_epi_plan();
  if (!pl) return GE_ERR_INVALID;
  st = read_majors(pl, opts);
  for (int g = 0; st == GE_OK && g < n_problems; ++g)
    st = check_alignment(pl, dtypes, problems[g].M, problems[g].N, problems[g].K);
  if (st != GE_OK) {
    delete pl;
    return st;
  }
  pl->n_groups = n_problems;
  pl->problems.assign(problems, problems + n_problems);
  pl->L = 1;
  pl->dt = *dtypes;
  pl->dag = *dag;
  if (opts) pl->opt = *opts;
  {
    const CompileResult cr = compile_program(*dtypes, *dag);
    st = cr.status;
    pl->prog = cr.prog;
  }
  if (st == GE_OK) {
    const bool interp = (pl->opt.debug_flags & GE_DEBUG_FORCE_INTERPRETER) != 0u;
    pl->epi = pick_executor(pl->prog, interp);
    pl->interp_epi = pl->prog.n_regs > 4 ? -2 : -1;
    st = check_device(&pl->device, &pl->num_sms, &pl->max_smem);
    if (st == GE_OK && pl->epi < 0 && !interp && pl->opt.specialize >= 0 && jit_available())
      pl->epi = kEpiSpecialized;
  }
  if (st == GE_OK) {
    void *sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_ge_status) != cudaSuccess) st = GE_ERR_CUDA;
    pl->status = static_cast<uint32_t *>(sym);
  }
  if (st == GE_OK) st = configure_grouped(pl);
  if (st == GE_ERR_JIT) {
    pl->epi = pl->interp_epi;
    st = configure_grouped(pl);
  }
  if (st == GE_OK && !encode_fn()) st = GE_ERR_CUDA;
  if (st == GE_OK) {
    const size_t bytes = sizeof(GroupDesc) * size_t(kGroupSlots) * size_t(n_problems);
    if (cudaMalloc(&pl->d_desc, bytes) != cudaSuccess ||
        cudaMallocHost(&pl->h_desc, bytes) != cudaSuccess)
      st = GE_ERR_CUDA;
    for (int s = 0; st == GE_OK && s < kGroupSlots; ++s)
      if (cudaEventCreateWithFlags(&pl->ev[s], cudaEventDisableTiming) != cudaSuccess)
        st = GE_ERR_CUDA;
  }
  if (st != GE_OK) {
    cudaGetLastError();
    delete pl;
    return st;
  }
  fill_group_shapes(pl);
  {
    const std::vector<int4> tiles = grouped_tile_table(pl);
    const size_t bytes = sizeof(int4) * tiles.size();
    if (cudaMalloc(&pl->d_tiles, bytes) != cudaSuccess ||
        cudaMemcpy(pl->d_tiles, tiles.data(), bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      delete pl;
      return GE_ERR_CUDA;
    }
  }
  fill_params(pl, pl->lay, pl->prog, &pl->kp);
  pl->kp.num_tiles = pl->lay.num_tiles;
  pl->kp.num_groups = n_problems;
  pl->kp.tile_info = pl->d_tiles;
  if (log_enabled()) log_plan(pl);
  *plan = pl;
  return GE_OK;
}

int gemm_epi_grouped_run(gemm_epi_plan *pl, const void *const *A, const void *const *B,
                         const void *const *aux, const float *scalars, void *const *outs,
                         void *stream) {
  if (!pl || !pl->n_groups) return GE_ERR_INVALID;
  int st = check_grouped_args(pl, A, B, aux, scalars, outs);
  if (st != GE_OK) return st;
  const int n = pl->n_groups, na = pl->dt.n_aux, no = pl->dt.n_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the pointers this run's table must hold
  std::vector<const void *> ptrs;
  ptrs.reserve(size_t(n) * (2 + na + no));
  for (int g = 0; g < n; ++g) {
    ptrs.push_back(A[g]);
    ptrs.push_back(B[g]);
    for (int a = 0; a < na; ++a) ptrs.push_back(aux ? aux[g * na + a] : nullptr);
    for (int o = 0; o < no; ++o) ptrs.push_back(outs[g * no + o]);
  }
  // the launch may overlap the previous kernel on the stream only when
  // nothing else precedes it: no table copy and no wait on another stream
  bool overlap = pl->opt.no_pdl == 0;
  if (pl->slot < 0 || pl->slot_ptrs[pl->slot] != ptrs) {
    overlap = false;
    const int next = (pl->slot + 1) % kGroupSlots;
    // the staging and device table of `next` are free once the run that used
    // them last has finished
    if (pl->ev_used[next] && cudaEventSynchronize(pl->ev[next]) != cudaSuccess) return GE_ERR_CUDA;
    pl->slot_ptrs[next].clear();
    if (!build_group_table(pl, next, A, B, aux, outs)) return GE_ERR_CUDA;
    const size_t bytes = sizeof(GroupDesc) * size_t(n);
    if (cudaMemcpyAsync(pl->d_desc + size_t(next) * n, pl->h_desc + size_t(next) * n, bytes,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return GE_ERR_CUDA;
    pl->slot = next;
    pl->slot_ptrs[next] = std::move(ptrs);
  } else if (pl->ev_used[pl->slot] && pl->ev_stream[pl->slot] != s) {
    // a table reused from another stream: order this run after the last run
    // that read it (which follows the table's copy), so every earlier reader
    // of the table is finished when its event next completes
    overlap = false;
    if (cudaStreamWaitEvent(s, pl->ev[pl->slot], 0) != cudaSuccess) return GE_ERR_CUDA;
  }
  KParams &kp = pl->kp;
  kp.groups = pl->d_desc + size_t(pl->slot) * n;
  for (int i = 0; i < pl->dt.n_scalar; ++i) kp.prog.scalars[i] = scalars[i];
  if (launch_gemm(pl->lay, pl->epi, kp, s, overlap) != cudaSuccess) return GE_ERR_CUDA;
  if (cudaEventRecord(pl->ev[pl->slot], s) != cudaSuccess) return GE_ERR_CUDA;
  pl->ev_used[pl->slot] = true;
  pl->ev_stream[pl->slot] = s;
  return GE_OK;
}

const char *gemm_epi_status_string(int status) {
  switch (status) {
    case GE_OK: return "GE_OK";
    case GE_ERR_NO_ACCUM: return "GE_ERR_NO_ACCUM";
    case GE_ERR_NO_D: return "GE_ERR_NO_D";
    case GE_ERR_SSA: return "GE_ERR_SSA";
    case GE_ERR_MISSING_ARG: return "GE_ERR_MISSING_ARG";
    case GE_ERR_UNSUPPORTED: return "GE_ERR_UNSUPPORTED";
    case GE_ERR_MISALIGNED: return "GE_ERR_MISALIGNED";
    case GE_ERR_ARCH: return "GE_ERR_ARCH";
    case GE_ERR_SHAPE: return "GE_ERR_SHAPE";
    case GE_ERR_TIMEOUT: return "GE_ERR_TIMEOUT";
    case GE_ERR_CUDA: return "GE_ERR_CUDA";
    case GE_ERR_INVALID: return "GE_ERR_INVALID";
    case GE_ERR_SMEM: return "GE_ERR_SMEM";
    case GE_ERR_WORKSPACE: return "GE_ERR_WORKSPACE";
    default: return "GE_ERR_UNKNOWN";
  }
}

int gemm_epi_last_error(gemm_epi_plan *plan) {
  (void)plan;
  uint32_t st[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(st, g_ge_status, sizeof(st)) != cudaSuccess) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  if (st[0] != 0) {
    const uint32_t zero[4] = {0, 0, 0, 0};
    if (log_enabled())
      std::fprintf(stderr, "[gemm_epi] device status %u (wait site %u, block %u)\n", st[0], st[1],
                   st[2]);
    if (cudaMemcpyToSymbol(g_ge_status, zero, sizeof(zero)) != cudaSuccess) {
      cudaGetLastError();
      return GE_ERR_CUDA;
    }
  }
  return static_cast<int>(st[0]);
}

}  // extern "C"

// ------------------------------------------------- allocation-free variant --
// The workspace of gemm_epi_run_unfused_noalloc: part of the library image, so
// every device that loads it holds these GE_NOALLOC_SCRATCH_BYTES until exit.
// In host code the name is only a stand-in for the symbol; the device address
// comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) float g_noalloc_scratch[GE_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

extern "C" int gemm_epi_run_unfused_noalloc(gemm_epi_plan *pl, const void *A, const void *B,
                                            const void *const *aux, const float *scalars,
                                            void *const *outs, void *stream) {
  if (!pl || pl->n_groups) return GE_ERR_INVALID;
  if (gemm_epi_unfused_workspace_bytes(pl) > GE_NOALLOC_SCRATCH_BYTES) return GE_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GE_ERR_CUDA;
  }
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
      // first call on this device (which is current): find the array's address
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return GE_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // The GEMM writes every workspace element before the elementwise kernel
  // reads it, so stale contents from an earlier call never leak through.
  return gemm_epi_run_unfused(pl, A, B, aux, scalars, outs, scratch, GE_NOALLOC_SCRATCH_BYTES,
                              stream);
}
