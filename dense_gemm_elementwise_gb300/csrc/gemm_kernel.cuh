// gemm_kernel.cuh -- persistent, warp-specialised GEMM + fused epilogue for sm_103a.
//
// The operation: "CUTLASS Operator API: Custom epilogue fusions for GEMMs"
// (the GEMM result accum goes through a user epilogue before anything is
// stored) and "Custom Epilogue Example", "Basic Example: Alpha-Beta Scaling"
// (the epilogue reads C and X tiles and writes D and Y in the same kernel).
// The pages' own kernel (128x128 MMA tile, 2x1 cluster, 2-CTA instructions,
// "Running the Example") is prior art for other hardware; the tiling here is
// this file's own.
//
// One CTA per SM (or one 2x1 cluster per SM pair with cta_group::2), looping
// over output tiles in a static round-robin order.  Warp roles:
//   warp 0      TMA producer: A and B k-blocks (K-major or MN-major) into an
//               S-stage shared-memory ring, full/empty mbarriers per stage.
//   warp 1      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma (fp16/bf16 -> fp32) into one of two TMEM
//               accumulators; tcgen05.commit frees ring stages and publishes
//               finished accumulators.
//   warps 2..   epilogue, 4 or 8 warps (Epi::kWarps; with 8, the two warps of
//               a TMEM lane quarter take alternate 32-column steps):
//               tcgen05.ld of 32-column steps, aux tensors staged per warp by
//               TMA (prefetched ahead, across tiles), the epilogue program in
//               fp32 (interpreted, or straight-line for catalog entries),
//               rounding, TMA stores from staging boxes.
// The two TMEM accumulators let the epilogue of tile i overlap the mainloop of
// tile i+1.  Ragged M/N/K edges are handled by TMA: out-of-range loads read
// zeros, out-of-range stores are dropped.  When the host splits the last wave
// (KParams::num_full), each of its tiles runs as two half-width tiles: MMA N
// = BN/2, half of each CTA's B atoms, half of the epilogue steps.
//
// A grouped launch (KParams::groups set) runs many problems of different
// sizes: tile t is looked up in a per-tile table (problem, m/n block, k
// blocks), and each problem brings its own tensor maps and vector pointers
// from a problem table in global memory.
//
// cta_group::2: the CTA pair computes a (256 x BN) tile.  Each CTA loads its
// 128 rows of A and its BN/2 columns of B into its own shared memory; the
// leader's MMA thread issues the pair MMA, which reads both CTAs' halves and
// writes each CTA's 128 accumulator rows into that CTA's TMEM.  Stage
// completion is counted on the leader's barriers; each commit arrives on the
// same barrier in both CTAs.  Every TMA load lands in the issuing CTA's own
// shared memory (no cluster multicast).
//
// Every wait is bounded (globaltimer): on expiry the kernel records
// GE_ERR_TIMEOUT in the status word, stops issuing work, waits (bounded) for
// its own copies in flight, frees TMEM and exits.
#pragma once

#include "common.cuh"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace ge {

template <int CG, int BN>
struct TileCfg {
  static constexpr int kCluster = CG;              // CTAs per cluster
  static constexpr int kMmaM = BM * CG;            // rows of one MMA tile
  static constexpr int kBnLocal = BN / CG;         // B columns loaded per CTA
  static constexpr int kABytes = BM * BK * 2;      // one A stage
  static constexpr int kBBytes = kBnLocal * BK * 2;
  static constexpr int kBAtoms = kBnLocal / 64;    // 64-column swizzle atoms of B
  static constexpr int kSteps = BN / EW;          // epilogue steps per tile
  static constexpr int kTmemCols = 2 * BN;         // two accumulators
  static_assert(kBnLocal % 64 == 0, "B half-tile must be whole 128-byte atoms");
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM alloc size");
};

// barrier block layout (bytes from off_bar)
constexpr uint32_t kBarFull = 0;                       // kMaxStages x 8
constexpr uint32_t kBarEmpty = 64;                     // kMaxStages x 8
constexpr uint32_t kBarTmemFull = 128;                 // 2 x 8
constexpr uint32_t kBarTmemEmpty = 144;                // 2 x 8
constexpr uint32_t kBarAux = 160;                      // kMaxEpiWarps x kMaxAuxStages x 8
constexpr uint32_t kBarDrain = kBarAux + 8 * kMaxEpiWarps * kMaxAuxStages;  // 672
constexpr uint32_t kTmemSlot = kBarDrain + 8;          // 680
constexpr uint32_t kAbortFlag = kTmemSlot + 4;         // 684
constexpr uint32_t kBarBlockBytes = 1024;
static_assert(kAbortFlag + 4 <= kBarBlockBytes, "barrier block overflow");

__device__ __forceinline__ void tile_coords(int num_m_blk, int num_n_blk, int G, int t, int &l,
                                            int &mb, int &nb) {
  const int per_batch = num_m_blk * num_n_blk;
  l = t / per_batch;
  const int r = t - l * per_batch;
  // raster: groups of G m-blocks; within a group m varies fastest, so tiles
  // processed at the same time share their B columns (and A rows across groups)
  const int group = r / (G * num_n_blk);
  const int first_m = group * G;
  const int gsize = min(num_m_blk - first_m, G);
  const int rr = r - group * G * num_n_blk;
  mb = first_m + rr % gsize;
  nb = rr / gsize;
}

// A tile of the launch: its batch and block coordinates, its k-block count,
// which column half it covers if it is half of a split tile and, for a
// grouped GEMM, the problem it belongs to.
struct TileRef {
  int l, mb, nb, num_kb;
  int half;             // -1: the whole BN columns; 0 / 1: the first / second BN/2
  const GroupDesc *gd;  // nullptr: the batched problem described by KParams
};

// Tile t of the launch: computed for a batched GEMM, one 16-byte table load
// for a grouped one.
__device__ __forceinline__ TileRef locate(const KParams &p, int t) {
  TileRef r;
  r.half = -1;
  if (p.groups == nullptr) {
    // tiles past num_full come in pairs: the two column halves of full tile
    // num_full + (t - num_full) / 2 (the last wave, split so that twice as
    // many CTAs share it)
    int tt = t;
    if (t >= p.num_full) {
      tt = p.num_full + ((t - p.num_full) >> 1);
      r.half = (t - p.num_full) & 1;
    }
    tile_coords(p.num_m_blk, p.num_n_blk, p.raster_group, tt, r.l, r.mb, r.nb);
    r.num_kb = p.num_kb;
    r.gd = nullptr;
  } else {
    const int4 ti = __ldg(p.tile_info + t);
    r.l = 0;
    r.mb = ti.y;
    r.nb = ti.z;
    r.num_kb = ti.w;
    r.gd = p.groups + ti.x;
  }
  return r;
}

// This CTA's tiles in order, each looked up one tile ahead so that a table
// load overlaps the work on the tile before it.
struct TileCursor {
  const KParams &p;
  int unit, n_units, count, i;
  TileRef nxt;
  __device__ __forceinline__ TileCursor(const KParams &p_, int unit_, int n_units_, int count_)
      : p(p_), unit(unit_), n_units(n_units_), count(count_), i(0) {
    if (count > 0) nxt = locate(p, unit);
  }
  __device__ __forceinline__ TileRef next() {
    const TileRef r = nxt;
    if (++i < count) nxt = locate(p, unit + i * n_units);
    return r;
  }
  // the tile after the one next() returned last (valid while i < count)
  __device__ __forceinline__ bool has_more() const { return i < count; }
};

struct Waiter {
  volatile uint32_t *abort_flag;  // shared: this CTA gave up
  uint32_t *status;               // global status block
  uint64_t timeout_ns;

  __device__ __forceinline__ void fail(uint32_t site) const {
    *abort_flag = 1u;
    if (atomicCAS(status, 0u, static_cast<uint32_t>(GE_ERR_TIMEOUT)) == 0u) {
      status[1] = site;
      status[2] = blockIdx.x;
    }
  }

  template <bool kCluster = false>
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, uint32_t site) const {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (kCluster ? mbar_try_wait_cluster(bar, parity)
                   : mbar_try_wait_sleep(bar, parity, 20000u))
        return true;
      if ((it & 3u) == 0u) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
          fail(site);
          return false;
        }
      }
    }
  }

  // teardown after an abort: ignores the abort flag, still bounded
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
      if (globaltimer_ns() - t0 > timeout_ns) {
        fail(SITE_DRAIN);
        return false;
      }
    }
    return true;
  }
};

// Epilogue leaves and stores for the fused kernel: aux tensors and outputs
// live in this warp's swizzled TMA staging boxes (row = lane, `half` picks the
// 16-column half of the 32-column box), broadcast vectors are read from
// global memory (the same addresses for every lane).
struct FusedMem {
  const KParams *p;
  const void *const *bptr;  // row-broadcast vectors of this tile's problem
  const void *const *cptr;  // column-broadcast vectors
  int M, N;                 // this tile's problem
  const uint8_t *aux_stage;
  uint8_t *out_stage;
  int row, half, col0;
  int grow;     // this lane's row within its batch (column-broadcast index)
  bool cd_m;    // staging boxes hold M-major tensors
  template <int DT>
  __device__ __forceinline__ void aux(uint32_t i, float (&t)[CH]) const {
    if (cd_m) col_box_load<DT>(aux_stage + p->aux_off[i], row, half, t);
    else box_load<DT>(aux_stage + p->aux_off[i], row, half, t);
  }
  template <int DT>
  __device__ __forceinline__ void bcast(uint32_t i, float (&t)[CH]) const {
    row_load<DT, CH>(bptr[i], col0, N, t);
  }
  template <int DT>
  __device__ __forceinline__ void cbcast(uint32_t i, float (&t)[CH]) const {
    const float v = grow < M ? load_one<DT>(cptr[i], grow) : 0.f;
#pragma unroll
    for (int e = 0; e < CH; ++e) t[e] = v;
  }
  template <int DT>
  __device__ __forceinline__ void store(uint32_t o, const float (&t)[CH]) const {
    if (cd_m) col_box_store<DT>(out_stage + p->out_off[o], row, half, t);
    else box_store<DT>(out_stage + p->out_off[o], row, half, t);
  }
};

template <int CG, int BN, class Epi>
__global__ void __launch_bounds__(threads_for(Epi::kWarps), 1)
    gemm_epi_kernel(const __grid_constant__ KParams p) {
  constexpr int kEpiWarps = Epi::kWarps;
  constexpr int kSplit = kEpiWarps / 4;  // warps per TMEM lane quarter
  static_assert(kEpiWarps == 4 || kEpiWarps == 8, "4 or 8 epilogue warps");
  using T = TileCfg<CG, BN>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the shared-window address (swizzle atoms)
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG > 1) ? cluster_ctarank() : 0u;  // rank within the CTA pair
  constexpr uint32_t leader = 0;             // cluster rank of the pair's leader
  const int unit = blockIdx.x / T::kCluster;  // this CTA's cluster (or CTA) index
  const int n_units = gridDim.x / T::kCluster;
  constexpr uint16_t kPairMask = 0x3u;  // a commit arrives in both CTAs of the pair

  const uint32_t bar = sb + p.off_bar;
  const uint32_t bar_aux = bar + kBarAux;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bar + kTmemSlot);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + p.off_bar + kAbortFlag);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar + kBarFull + 8 * s, 1);
      mbar_init(bar + kBarEmpty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar + kBarTmemFull + 8 * b, 1);
      mbar_init(bar + kBarTmemEmpty + 8 * b, kEpiWarps * CG);
    }
    for (int i = 0; i < kEpiWarps * kMaxAuxStages; ++i) mbar_init(bar_aux + 8 * i, 1);
    mbar_init(bar + kBarDrain, 1);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0 && p.groups == nullptr) {
    prefetch_tensormap(&p.tmA);
    prefetch_tensormap(&p.tmB);
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), T::kTmemCols);
    tmem_relinquish<CG>();
  }
  __syncwarp();
  tc_fence_before();
  if constexpr (T::kCluster > 1) cluster_sync_all(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
  const Waiter wt{abort_flag, p.status, p.timeout_ns};
  const int my_tiles = unit < p.num_tiles ? (p.num_tiles - 1 - unit) / n_units + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0, skipped = -1;
      bool skip = (p.debug_flags & GE_DEBUG_SKIP_FIRST_LOAD) != 0u;
      bool ok = true;
      TileCursor tc(p, unit, n_units, my_tiles);
      const GroupDesc *ready_gd = nullptr;  // problem whose A/B maps are fenced and prefetched
      for (int i = 0; ok && i < my_tiles; ++i) {
        const TileRef tr = tc.next();
        const int l = tr.l, mb = tr.mb, nb = tr.nb;
        const CUtensorMap *mA = tr.gd ? &tr.gd->tmA : &p.tmA;
        const CUtensorMap *mB = tr.gd ? &tr.gd->tmB : &p.tmB;
        if (tr.gd && tr.gd != ready_gd) {
          fence_tensormap_acquire(mA);
          fence_tensormap_acquire(mB);
          ready_gd = tr.gd;
        }
        const int m0 = mb * T::kMmaM + static_cast<int>(rank) * BM;
        // a half tile: BN/2 columns, BN/(2 CG) of them (half the B atoms) per CTA
        const bool half = tr.half >= 0;
        const int n0 = nb * BN + (tr.half > 0 ? BN / 2 : 0) +
                       static_cast<int>(rank) * (half ? T::kBnLocal / 2 : T::kBnLocal);
        const int b_atoms = half ? T::kBAtoms / 2 : T::kBAtoms;
        const uint32_t tx = half ? p.tx_bytes_half : p.tx_bytes;
        for (int kb = 0; kb < tr.num_kb; ++kb) {
          if (!wt.wait(bar + kBarEmpty + 8 * stage, phase ^ 1u, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          // k-snake: a CTA's odd tiles (every CTA is on its i-th tile during
          // wave i) walk K backwards, so a wave starts on the k slices the
          // wave before it loaded last, still in L2 (8192^3: 10 % fewer
          // DRAM reads).  Tiles of one wave still walk K in step, sharing
          // each slice's DRAM read.  The MMA order is the k order issued
          // (the first issued k-block starts the accumulator).
          const int kx = ((i & 1) ? tr.num_kb - 1 - kb : kb) * BK;
          if (skip) {
            skip = false;
            skipped = fills;
          } else {
            const uint32_t fb_local = bar + kBarFull + 8 * stage;
            const uint32_t sa = sb + p.off_A + stage * T::kABytes;
            const uint32_t sbb = sb + p.off_B + stage * T::kBBytes;
            if constexpr (CG == 2) {
              const uint32_t fb = mapa_shared(fb_local, leader);
              if (rank == 0) mbar_arrive_expect_tx(fb_local, tx);
              if (p.a_mn) {  // two 64-row atoms of the M-major A tile
                tma_load_3d_pair(sa, mA, fb, m0, kx, l);
                tma_load_3d_pair(sa + 8192, mA, fb, m0 + 64, kx, l);
              } else {
                tma_load_3d_pair(sa, mA, fb, kx, m0, l);
              }
              if (p.b_k) {
                tma_load_3d_pair(sbb, mB, fb, kx, n0, l);
              } else {
#pragma unroll
                for (int j = 0; j < T::kBAtoms; ++j)
                  if (j < b_atoms) tma_load_3d_pair(sbb + j * 8192, mB, fb, n0 + 64 * j, kx, l);
              }
            } else {
              mbar_arrive_expect_tx(fb_local, tx);
              if (p.a_mn) {
                tma_load_3d(sa, mA, fb_local, m0, kx, l);
                tma_load_3d(sa + 8192, mA, fb_local, m0 + 64, kx, l);
              } else {
                tma_load_3d(sa, mA, fb_local, kx, m0, l);
              }
              if (p.b_k) {
                tma_load_3d(sbb, mB, fb_local, kx, n0, l);
              } else {
#pragma unroll
                for (int j = 0; j < T::kBAtoms; ++j)
                  if (j < b_atoms) tma_load_3d(sbb + j * 8192, mB, fb_local, n0 + 64 * j, kx, l);
              }
            }
          }
          ++fills;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        // while the MMA drains this tile, make the next problem's maps ready
        if (tc.has_more() && tc.nxt.gd && tc.nxt.gd != ready_gd) {
          ready_gd = tc.nxt.gd;
          fence_tensormap_acquire(&ready_gd->tmA);
          fence_tensormap_acquire(&ready_gd->tmB);
          prefetch_tensormap(&ready_gd->tmA);
          prefetch_tensormap(&ready_gd->tmB);
        }
      }
      if (ok) {
        // tail: every stage released by the MMA, so all commit arrivals landed
        for (int i = 0; i < p.stages; ++i) {
          if (!wt.wait(bar + kBarEmpty + 8 * stage, phase ^ 1u, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && rank == 0) {
        // abort: wait for the copies still in flight into this CTA pair
        for (int f = fills - p.stages; f < fills; ++f) {
          if (f < 0 || f == skipped) continue;
          wt.drain(bar + kBarFull + 8 * (f % p.stages), static_cast<uint32_t>(f / p.stages) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0 && rank == 0) {
      const uint32_t id = make_idesc_f16(p.ab_bf16 != 0, T::kMmaM, BN, p.a_mn != 0, p.b_k == 0);
      const uint32_t id_half = make_idesc_f16(p.ab_bf16 != 0, T::kMmaM, BN / 2, p.a_mn != 0, p.b_k == 0);
      // per-k step advance and strides of the two operands' smem descriptors:
      // K-major tiles are 128-byte rows (k step 32 bytes, 8-row groups 1 KiB
      // apart), MN-major tiles are 64-element atoms 8 KiB apart whose k rows
      // are 128 bytes (k step 16 rows = 2 KiB).  The descriptors of stage 0 are
      // built once; a stage or k step only moves the start address, whose
      // field (address >> 4, bits 0-13) is added to directly: shared-memory
      // addresses stay below 256 KiB, so the sum never carries out of it.
      // This keeps the issuing thread to a few adds per MMA, well ahead of
      // the tensor pipe.
      const uint32_t a_step = p.a_mn ? 2048u : 32u, a_lbo = p.a_mn ? 8192u : 16u;
      const uint32_t b_step = p.b_k ? 32u : 2048u, b_lbo = p.b_k ? 16u : p.b_lbo;
      const uint32_t b_sbo = p.b_k ? 1024u : p.b_sbo;
      const uint64_t a_desc0 = smem_desc_sw128(sb + p.off_A, a_lbo, 1024u);
      const uint64_t b_desc0 = smem_desc_sw128(sb + p.off_B, b_lbo, b_sbo);
      const uint32_t a_k16 = a_step >> 4, b_k16 = b_step >> 4;
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      bool ok = true;
      TileCursor tc(p, unit, n_units, my_tiles);
      for (int i = 0; ok && i < my_tiles; ++i) {
        const TileRef tr = tc.next();
        const int num_kb = tr.num_kb;
        const uint32_t idt = tr.half < 0 ? id : id_half;
        if (!wt.wait<CG == 2>(bar + kBarTmemEmpty + 8 * abuf, aphase ^ 1u, SITE_MMA_TMEM_EMPTY)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(abuf * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wt.wait(bar + kBarFull + 8 * stage, phase, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage * (T::kABytes >> 4));
          const uint64_t bd = b_desc0 + static_cast<uint32_t>(stage * (T::kBBytes >> 4));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_f16<CG>(d, ad + a_k16 * k, bd + b_k16 * k, idt, (kb | k) != 0 ? 1u : 0u);
          umma_commit<CG>(bar + kBarEmpty + 8 * stage, kPairMask);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit<CG>(bar + kBarTmemFull + 8 * abuf, kPairMask);
        abuf ^= 1;
        if (abuf == 0) aphase ^= 1u;
      }
      if (ok) {
        // tail: both accumulators released, so every epilogue arrival landed
        for (int i = 0; i < 2; ++i) {
          if (!wt.wait<CG == 2>(bar + kBarTmemEmpty + 8 * abuf, aphase ^ 1u, SITE_MMA_TMEM_EMPTY))
            break;
          abuf ^= 1;
          if (abuf == 0) aphase ^= 1u;
        }
      } else {
        // abort: let the MMAs already issued finish before TMEM is freed
        umma_commit<CG>(bar + kBarDrain, kPairMask);
        wt.drain(bar + kBarDrain, 0u);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int e = warp - 2;  // staging slot
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ch = e / 4;    // which of the quarter's warps: takes steps ch, ch + kSplit, ...
    constexpr int kStepsW = T::kSteps / kSplit;  // this warp's steps per tile
    static_assert(T::kSteps % kSplit == 0, "steps split evenly between a quarter's warps");
    // a half tile has half the steps (the host splits tiles only where that
    // is a whole, nonzero number per warp)
    constexpr int kHalfW = kStepsW / 2 > 0 ? kStepsW / 2 : 1;
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t *aux_w = smem + p.off_aux + e * p.aux_stages * p.aux_stage_bytes;
    constexpr int kOutBufs = out_bufs_for(kEpiWarps);
    uint8_t *out_w = smem + p.off_out + e * kOutBufs * p.out_stage_bytes;
    const uint32_t auxbar_w = bar_aux + 8u * e * kMaxAuxStages;
    const bool has_aux = p.prog.n_tma_aux > 0;
    const int SA = p.aux_stages;
    // this CTA's full tiles come first, then its half tiles
    const int q_full = unit < p.num_full ? min((p.num_full - 1 - unit) / n_units + 1, my_tiles) : 0;
    const int full_steps = q_full * kStepsW;
    const int total = full_steps + (my_tiles - q_full) * kHalfW;
    int issued = 0, g = 0, abuf = 0, obuf = 0;
    uint32_t aphase = 0;
    bool ok = true;
    int pf_tile = -1, pf_x0 = 0, pf_y = 0, pf_l = 0;  // prefetch: coordinates of tile pf_tile
    TileCursor pf_tc(p, unit, n_units, my_tiles);        // tiles of the aux prefetch
    TileCursor tc(p, unit, n_units, my_tiles);           // tiles of the epilogue proper
    const CUtensorMap *pf_maps = p.tmAux;               // aux maps of tile pf_tile
    const GroupDesc *out_gd = nullptr;                  // problem whose output maps are fenced

    // TMA loads of every Load tensor for this warp's 32 rows of step gi
    auto issue_aux = [&](int gi) {
      const int ii = gi < full_steps ? gi / kStepsW : q_full + (gi - full_steps) / kHalfW;
      const int first = ii <= q_full ? ii * kStepsW : full_steps + (ii - q_full) * kHalfW;
      if (ii != pf_tile) {
        const TileRef tr = pf_tc.next();  // tiles are entered in order, one at a time
        pf_l = tr.l;
        pf_tile = ii;
        pf_x0 = tr.nb * BN + (tr.half > 0 ? BN / 2 : 0);
        pf_y = tr.mb * T::kMmaM + static_cast<int>(rank) * BM + q * 32;
        if (tr.gd && pf_maps != tr.gd->tmAux)
          for (int a = 0; a < p.prog.n_tma_aux; ++a) {
            fence_tensormap_acquire(&tr.gd->tmAux[a]);
            prefetch_tensormap(&tr.gd->tmAux[a]);
          }
        pf_maps = tr.gd ? tr.gd->tmAux : p.tmAux;
      }
      const int as = gi % SA;
      const uint32_t ab = auxbar_w + 8u * as;
      uint8_t *dst = aux_w + as * p.aux_stage_bytes;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(ab, p.aux_tx_bytes);
      const int x = pf_x0 + ((gi - first) * kSplit + ch) * EW;
      for (int a = 0; a < p.prog.n_tma_aux; ++a)
        tma_load_3d(smem_u32(dst + p.aux_off[a]), &pf_maps[a], ab, p.cd_m ? pf_y : x,
                    p.cd_m ? x : pf_y, pf_l);
    };

    for (int i = 0; ok && i < my_tiles; ++i) {
      const TileRef tr = tc.next();
      const int l = tr.l, mb = tr.mb, nb = tr.nb;
      const int m0 = mb * T::kMmaM + static_cast<int>(rank) * BM + q * 32;
      const int n0 = nb * BN + (tr.half > 0 ? BN / 2 : 0);
      const int steps = tr.half < 0 ? T::kSteps : T::kSteps / 2;  // 32-column steps of this tile
      const CUtensorMap *out_maps = tr.gd ? tr.gd->tmOut : p.tmOut;
      const void *const *bptr = tr.gd ? tr.gd->bcast_ptr : p.bcast_ptr;
      const void *const *cptr = tr.gd ? tr.gd->cbcast_ptr : p.cbcast_ptr;
      const int pM = tr.gd ? __ldg(&tr.gd->M) : p.M;
      const int pN = tr.gd ? __ldg(&tr.gd->N) : p.N;
      // output maps of this problem, unless made ready during the last tile
      if (lane == 0 && tr.gd && tr.gd != out_gd) {
        for (int o = 0; o < p.prog.n_out; ++o) fence_tensormap_acquire(&out_maps[o]);
        out_gd = tr.gd;
      }
      // start this tile's aux loads before its accumulator is ready
      if (has_aux && lane == 0) {
        while (issued < total && issued < g + SA) issue_aux(issued++);
      }
      __syncwarp();
      const bool got = wt.wait(bar + kBarTmemFull + 8 * abuf, aphase, SITE_EPI_TMEM_FULL);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      // the next tile's problem: make its output maps ready while this tile's
      // epilogue runs (its table entry was loaded with this tile's)
      if (lane == 0 && tc.has_more() && tc.nxt.gd && tc.nxt.gd != out_gd) {
        out_gd = tc.nxt.gd;
        for (int o = 0; o < p.prog.n_out; ++o) {
          fence_tensormap_acquire(&out_gd->tmOut[o]);
          prefetch_tensormap(&out_gd->tmOut[o]);
        }
      }
      tc_fence_after();
      for (int s = ch; s < steps; s += kSplit, ++g) {
        if (has_aux && lane == 0) {
          while (issued < total && issued < g + SA) issue_aux(issued++);
        }
        __syncwarp();
        float acc0[CH], acc1[CH];
        const uint32_t col = static_cast<uint32_t>(abuf * BN + s * EW);
        tmem_ld16(tq + col, acc0);
        tmem_ld16(tq + col + CH, acc1);
        tmem_wait_ld();
        if (s + kSplit >= steps) {
          // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            const uint32_t tb = bar + kBarTmemEmpty + 8 * abuf;
            if constexpr (CG == 2) mbar_arrive_remote(mapa_shared(tb, leader));
            else mbar_arrive(tb);
          }
        }
        if (has_aux) {
          const bool a_ok = wt.wait(auxbar_w + 8u * (g % SA), static_cast<uint32_t>(g / SA) & 1u,
                                    SITE_EPI_AUX_FULL);
          if (!__all_sync(0xffffffffu, a_ok)) {
            ok = false;
            break;
          }
        }
        // the staging buffer about to be written has been read by its last store
        if (lane == 0) bulk_wait_group_read<kOutBufs - 1>();
        __syncwarp();
        uint8_t *ostage = out_w + obuf * p.out_stage_bytes;
        const uint8_t *astage = aux_w + (g % SA) * p.aux_stage_bytes;
        const int c0 = n0 + s * EW;
        Epi::template run<CH>(p.prog, acc0, FusedMem{&p, bptr, cptr, pM, pN, astage, ostage, lane,
                                                     0, c0, m0 + lane, p.cd_m != 0});
        Epi::template run<CH>(p.prog, acc1, FusedMem{&p, bptr, cptr, pM, pN, astage, ostage, lane,
                                                     1, c0 + CH, m0 + lane, p.cd_m != 0});
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int o = 0; o < p.prog.n_out; ++o)
            tma_store_3d(&out_maps[o], smem_u32(ostage + p.out_off[o]), p.cd_m ? m0 : c0,
                         p.cd_m ? c0 : m0, l);
          bulk_commit_group();
        }
        if constexpr (kOutBufs == 2) obuf ^= 1;
      }
      abuf ^= 1;
      if (abuf == 0) aphase ^= 1u;
    }
    if (lane == 0) {
      if (!ok)
        for (int gi = g; gi < issued; ++gi)
          wt.drain(auxbar_w + 8u * (gi % SA), static_cast<uint32_t>(gi / SA) & 1u);
      bulk_wait_group<0>();
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown --
  __syncwarp();
  tc_fence_before();
  if constexpr (T::kCluster > 1) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, T::kTmemCols);
  }
}

}  // namespace ge
