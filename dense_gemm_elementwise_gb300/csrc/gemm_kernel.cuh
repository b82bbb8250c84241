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
//   warp 2      epilogue TMA thread: for every 32-column step of every tile
//               it loads each aux tensor's 128-row x 32-column box (all of
//               this CTA's accumulator rows) into a staging slot ahead of
//               time, and stores each output's box once the epilogue warps
//               have written it.  One thread issues every epilogue copy, a
//               quarter as many as 32-row boxes would take, and the
//               epilogue warps never wait on a copy being issued.
//   warps 3..   epilogue, one or two groups of 4 warps (Epi::kWarps 4 or 8;
//               a group's warps cover the four TMEM lane quarters, and two
//               groups take alternate 32-column steps): tcgen05.ld of the
//               step, the epilogue program in fp32 (interpreted, or
//               straight-line for catalog entries) on the staged aux boxes,
//               rounding into the output staging box.  Slots and boxes are
//               handed over through mbarriers (aux full / empty, out full /
//               empty).
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
// epilogue staging, per warp group and slot (group-major)
constexpr uint32_t kBarAuxFull = 160;                  // kMaxEpiGroups x kMaxAuxStages x 8
constexpr uint32_t kBarAuxEmpty = kBarAuxFull + 8 * kMaxEpiGroups * kMaxAuxStages;  // 288
constexpr uint32_t kBarOutFull = kBarAuxEmpty + 8 * kMaxEpiGroups * kMaxAuxStages;  // 416
constexpr uint32_t kBarOutEmpty = kBarOutFull + 8 * kMaxEpiGroups * kMaxOutBufs;    // 448
constexpr uint32_t kBarDrain = kBarOutEmpty + 8 * kMaxEpiGroups * kMaxOutBufs;      // 480
constexpr uint32_t kTmemSlot = kBarDrain + 8;          // 488
constexpr uint32_t kAbortFlag = kTmemSlot + 4;         // 492
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
// live in the warp group's swizzled 128-row TMA staging boxes (row = the
// lane's accumulator row, 32 * quarter + lane; `half` picks the 16-column
// half of the 32-column box), broadcast vectors are read from global memory
// (the same addresses for every lane).
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
  constexpr int kGroups = kEpiWarps / 4;      // epilogue warp groups
  constexpr int kOutBufs = out_bufs_for(kEpiWarps);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bar + kTmemSlot);
  volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + p.off_bar + kAbortFlag);

  if (warp == 0) {
    // the lanes of warp 0 initialise the barriers in parallel
    if (lane < p.stages) {
      mbar_init(bar + kBarFull + 8 * lane, 1);
      mbar_init(bar + kBarEmpty + 8 * lane, 1);
    }
    if (lane < 2) {
      mbar_init(bar + kBarTmemFull + 8 * lane, 1);
      mbar_init(bar + kBarTmemEmpty + 8 * lane, kEpiWarps * CG);
    }
    if (lane < kGroups * kMaxAuxStages) {  // slot (lane % kMaxAuxStages) of group (lane / ...)
      mbar_init(bar + kBarAuxFull + 8 * lane, 1);
      mbar_init(bar + kBarAuxEmpty + 8 * lane, 4);  // the group's 4 warps release a slot
    }
    if (lane < kGroups * kMaxOutBufs) {
      mbar_init(bar + kBarOutFull + 8 * lane, 4);   // the group's 4 warps fill a box
      mbar_init(bar + kBarOutEmpty + 8 * lane, 1);  // the TMA thread frees it
    }
    if (lane == 0) {
      mbar_init(bar + kBarDrain, 1);
      *abort_flag = 0u;
    }
    fence_mbarrier_init();
    __syncwarp();
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
  // Launched with programmatic stream serialization, this grid may start
  // while the previous kernel on the stream is still running: the set-up
  // above touches no global memory; every role waits here before its first
  // read of an input or write of an output.
  griddep_wait();
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
      // every operand copy is issued: the next launch on the stream may be
      // scheduled (its CTAs start as SMs free up and wait for this grid)
      griddep_launch_dependents();
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
  } else if (warp == 2) {
    // ------------------------------------------------- epilogue TMA thread --
    // Walks this CTA's tiles and their 32-column steps twice, as two
    // sequences: the aux loads (step g of a group into slot g % SA, once the
    // group has released it) run ahead of the output stores (step g's boxes,
    // once the group's four warps have filled them).  One polling loop
    // serves both, so neither blocks the other.
    if (lane == 0) {
      const bool has_aux = p.prog.n_tma_aux > 0;
      const int SA = p.aux_stages;
      TileCursor ltc(p, unit, n_units, my_tiles), stc(p, unit, n_units, my_tiles);
      int l_i = 0, l_s = 0, l_steps = 0, l_x0 = 0, l_y0 = 0, l_l = 0;
      int s_i = 0, s_s = 0, s_steps = 0, s_x0 = 0, s_y0 = 0, s_l = 0;
      int l_g[kMaxEpiGroups] = {0, 0}, s_g[kMaxEpiGroups] = {0, 0};
      const CUtensorMap *l_maps = p.tmAux, *s_maps = p.tmOut;
      const GroupDesc *l_gd = nullptr, *s_gd = nullptr;  // problems whose maps are fenced
      bool l_more = has_aux && my_tiles > 0, s_more = my_tiles > 0;
      // a tile's column origin, this CTA's first accumulator row, batch, steps
      auto enter = [&](const TileRef &tr, int &x0, int &y0, int &ll, int &steps) {
        x0 = tr.nb * BN + (tr.half > 0 ? BN / 2 : 0);
        y0 = tr.mb * T::kMmaM + static_cast<int>(rank) * BM;
        ll = tr.l;
        steps = tr.half < 0 ? T::kSteps : T::kSteps / 2;
      };
      if (l_more) {
        const TileRef tr = ltc.next();
        enter(tr, l_x0, l_y0, l_l, l_steps);
        if (tr.gd) {
          l_gd = tr.gd;
          l_maps = tr.gd->tmAux;
          for (int a = 0; a < p.prog.n_tma_aux; ++a) fence_tensormap_acquire(&l_maps[a]);
        }
      }
      if (s_more) {
        const TileRef tr = stc.next();
        enter(tr, s_x0, s_y0, s_l, s_steps);
        if (tr.gd) {
          s_gd = tr.gd;
          s_maps = tr.gd->tmOut;
          for (int o = 0; o < p.prog.n_out; ++o) fence_tensormap_acquire(&s_maps[o]);
        }
      }
      uint64_t t_idle = globaltimer_ns();
      uint32_t polls = 0;
      bool ok = true;
      while (ok && (l_more || s_more)) {
        bool progress = false;
        if (s_more) {
          const int grp = s_s % kGroups;
          const int buf = s_g[grp] % kOutBufs;
          const uint32_t fb = bar + kBarOutFull + 8u * (grp * kMaxOutBufs + buf);
          if (mbar_test_wait(fb, static_cast<uint32_t>(s_g[grp] / kOutBufs) & 1u)) {
            const uint8_t *box = smem + p.off_out + (grp * kOutBufs + buf) * p.out_stage_bytes;
            const int x = s_x0 + s_s * EW;
            for (int o = 0; o < p.prog.n_out; ++o)
              tma_store_3d(&s_maps[o], smem_u32(box + p.out_off[o]), p.cd_m ? s_y0 : x,
                           p.cd_m ? x : s_y0, s_l);
            bulk_commit_group();
            // the box is free once the copy has read it
            bulk_wait_group_read<0>();
            mbar_arrive(bar + kBarOutEmpty + 8u * (grp * kMaxOutBufs + buf));
            ++s_g[grp];
            if (++s_s == s_steps) {
              s_s = 0;
              if (++s_i < my_tiles) {
                const TileRef tr = stc.next();
                enter(tr, s_x0, s_y0, s_l, s_steps);
                if (tr.gd) {
                  s_maps = tr.gd->tmOut;
                  if (tr.gd != s_gd) {
                    s_gd = tr.gd;
                    for (int o = 0; o < p.prog.n_out; ++o) fence_tensormap_acquire(&s_maps[o]);
                  }
                }
              } else {
                s_more = false;
              }
            }
            progress = true;
          }
        }
        if (l_more) {
          const int grp = l_s % kGroups;
          const int slot = l_g[grp] % SA;
          const uint32_t eb = bar + kBarAuxEmpty + 8u * (grp * kMaxAuxStages + slot);
          if (mbar_test_wait(eb, (static_cast<uint32_t>(l_g[grp] / SA) & 1u) ^ 1u)) {
            const uint32_t fb = bar + kBarAuxFull + 8u * (grp * kMaxAuxStages + slot);
            const uint8_t *box = smem + p.off_aux + (grp * SA + slot) * p.aux_stage_bytes;
            const int x = l_x0 + l_s * EW;
            mbar_arrive_expect_tx(fb, p.aux_tx_bytes);
            for (int a = 0; a < p.prog.n_tma_aux; ++a)
              tma_load_3d(smem_u32(box + p.aux_off[a]), &l_maps[a], fb, p.cd_m ? l_y0 : x,
                          p.cd_m ? x : l_y0, l_l);
            ++l_g[grp];
            if (++l_s == l_steps) {
              l_s = 0;
              if (++l_i < my_tiles) {
                const TileRef tr = ltc.next();
                enter(tr, l_x0, l_y0, l_l, l_steps);
                if (tr.gd) {
                  l_maps = tr.gd->tmAux;
                  if (tr.gd != l_gd) {
                    l_gd = tr.gd;
                    for (int a = 0; a < p.prog.n_tma_aux; ++a) {
                      fence_tensormap_acquire(&l_maps[a]);
                      prefetch_tensormap(&l_maps[a]);
                    }
                  }
                }
              } else {
                l_more = false;
              }
            }
            progress = true;
          }
        }
        if (progress) {
          t_idle = globaltimer_ns();
          polls = 0;
        } else if ((++polls & 15u) == 0u) {
          if (*abort_flag) {
            ok = false;
          } else if (globaltimer_ns() - t_idle > p.timeout_ns) {
            wt.fail(SITE_EPI_TMA);
            ok = false;
          } else {
            __nanosleep(64);
          }
        }
      }
      if (!ok) {
        // abort: wait (bounded) for the aux loads still in flight, the last
        // one issued into each slot
        for (int grp = 0; grp < kGroups; ++grp)
          for (int j = max(l_g[grp] - SA, 0); j < l_g[grp]; ++j)
            wt.drain(bar + kBarAuxFull + 8u * (grp * kMaxAuxStages + j % SA),
                     static_cast<uint32_t>(j / SA) & 1u);
      }
      bulk_wait_group<0>();
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int e = warp - kEpiWarp0;  // epilogue warp index
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int grp = e / 4;           // group: takes steps grp, grp + kGroups, ...
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const bool has_aux = p.prog.n_tma_aux > 0;
    const int SA = p.aux_stages;
    const int row = q * 32 + lane;   // this lane's row of the CTA's 128 accumulator rows
    int g = 0, abuf = 0;             // this group's steps so far
    uint32_t aphase = 0;
    bool ok = true;
    TileCursor tc(p, unit, n_units, my_tiles);

    for (int i = 0; ok && i < my_tiles; ++i) {
      const TileRef tr = tc.next();
      const int m0 = tr.mb * T::kMmaM + static_cast<int>(rank) * BM + q * 32;
      const int n0 = tr.nb * BN + (tr.half > 0 ? BN / 2 : 0);
      const int steps = tr.half < 0 ? T::kSteps : T::kSteps / 2;  // 32-column steps of this tile
      const void *const *bptr = tr.gd ? tr.gd->bcast_ptr : p.bcast_ptr;
      const void *const *cptr = tr.gd ? tr.gd->cbcast_ptr : p.cbcast_ptr;
      const int pM = tr.gd ? __ldg(&tr.gd->M) : p.M;
      const int pN = tr.gd ? __ldg(&tr.gd->N) : p.N;
      const bool got = wt.wait(bar + kBarTmemFull + 8 * abuf, aphase, SITE_EPI_TMEM_FULL);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int s = grp; s < steps; s += kGroups, ++g) {
        float acc0[CH], acc1[CH];
        const uint32_t col = static_cast<uint32_t>(abuf * BN + s * EW);
        tmem_ld16(tq + col, acc0);
        tmem_ld16(tq + col + CH, acc1);
        tmem_wait_ld();
        if (s + kGroups >= steps) {
          // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            const uint32_t tb = bar + kBarTmemEmpty + 8 * abuf;
            if constexpr (CG == 2) mbar_arrive_remote(mapa_shared(tb, leader));
            else mbar_arrive(tb);
          }
        }
        const int slot = g % SA, buf = g % kOutBufs;
        if (has_aux) {
          const bool a_ok = wt.wait(bar + kBarAuxFull + 8u * (grp * kMaxAuxStages + slot),
                                    static_cast<uint32_t>(g / SA) & 1u, SITE_EPI_AUX_FULL);
          if (!__all_sync(0xffffffffu, a_ok)) {
            ok = false;
            break;
          }
        }
        // the output box about to be written has been read by its last store
        const bool o_ok = wt.wait(bar + kBarOutEmpty + 8u * (grp * kMaxOutBufs + buf),
                                  (static_cast<uint32_t>(g / kOutBufs) & 1u) ^ 1u,
                                  SITE_EPI_OUT_EMPTY);
        if (!__all_sync(0xffffffffu, o_ok)) {
          ok = false;
          break;
        }
        uint8_t *ostage = smem + p.off_out + (grp * kOutBufs + buf) * p.out_stage_bytes;
        const uint8_t *astage = smem + p.off_aux + (grp * SA + slot) * p.aux_stage_bytes;
        const int c0 = n0 + s * EW;
        Epi::template run<CH>(p.prog, acc0, FusedMem{&p, bptr, cptr, pM, pN, astage, ostage, row,
                                                     0, c0, m0 + lane, p.cd_m != 0});
        Epi::template run<CH>(p.prog, acc1, FusedMem{&p, bptr, cptr, pM, pN, astage, ostage, row,
                                                     1, c0 + CH, m0 + lane, p.cd_m != 0});
        // the aux slot has been read; the output box is written (visible to
        // the TMA engine after the proxy fence)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (has_aux) mbar_arrive(bar + kBarAuxEmpty + 8u * (grp * kMaxAuxStages + slot));
          mbar_arrive(bar + kBarOutFull + 8u * (grp * kMaxOutBufs + buf));
        }
      }
      abuf ^= 1;
      if (abuf == 0) aphase ^= 1u;
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
