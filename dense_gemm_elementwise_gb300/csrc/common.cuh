// common.cuh -- definitions shared by the host plan and the sm_103a kernels:
// the compiled epilogue program and the kernel parameter block.
#pragma once

#include "gemm_epi.h"

#ifdef __CUDACC_RTC__
// compiled at run time (kernels specialised for one epilogue program): the
// tensor-map type with the driver header's size and alignment
typedef struct CUtensorMap_st {
  alignas(128) unsigned long long opaque[16];
} CUtensorMap;
#else
#include <cuda.h>  // CUtensorMap (type only; the driver is reached through cudart)
#include <stdint.h>
#endif

namespace ge {

// ---------------------------------------------------------------------------
// Epilogue program.
//
// The host compiles the ge_dag into a short two-address program over a few
// fp32 vector registers, each holding CH consecutive columns of one output
// row (a thread's share of an epilogue chunk).  Leaves of the DAG (the
// accumulator, aux tensors, row-broadcast vectors, scalars) are read straight
// from their source by the instruction that consumes them, so the program
// only materialises intermediate values.  The interpreter loops over
// instructions outside and over the CH columns inside: dispatch is paid once
// per instruction per chunk, not per element.
// ---------------------------------------------------------------------------
constexpr int CH = 16;        // columns one program evaluation covers per thread
constexpr int EW = 32;        // columns of one fused-epilogue step (TMA box width)
constexpr int kRegs = 8;      // vector registers of the epilogue program (at most)
constexpr int kMaxIns = 48;   // instructions in one program

enum EpiOp : uint32_t {
  OP_MOV = 0,    // r[dst]  = src
  OP_MUL = 1,    // r[dst] *= src
  OP_ADD = 2,    // r[dst] += src
  OP_RELU = 3,   // r[dst]  = r[dst] > 0 ? r[dst] : +0
  OP_STORE = 4,  // out[dst] = round(src)
  OP_SUB = 5,    // r[dst] -= src
  OP_RSUB = 6,   // r[dst]  = src - r[dst]
  OP_DIV = 7,    // r[dst] /= src
  OP_RDIV = 8,   // r[dst]  = src / r[dst]
  OP_MIN = 9,    // r[dst]  = min(r[dst], src)
  OP_MAX = 10,   // r[dst]  = max(r[dst], src)
  // activations read their operand from any source: r[dst] = f(src)
  OP_SIGMOID = 11,
  OP_TANH = 12,
  OP_GELU = 13,
  OP_SILU = 14,
  OP_HARDSWISH = 15,
  OP_LEAKY = 16,   // r[dst]  = r[dst] > 0 ? r[dst] : src * r[dst]   (src: slope)
  OP_RLEAKY = 17,  // r[dst]  = src > 0 ? src : r[dst] * src         (r[dst]: slope)
};

enum EpiSrc : uint32_t {
  SRC_REG = 0,     // r[idx]
  SRC_ACC = 1,     // accumulator
  SRC_AUX = 2,     // Load tensor number idx (TMA-staged in the fused kernel)
  SRC_BCAST = 3,   // row-broadcast vector number idx
  SRC_SCALAR = 4,  // scalar idx
  SRC_NONE = 5,
  SRC_CBCAST = 6,  // column-broadcast vector number idx (one value per row)
};

__host__ __device__ constexpr uint32_t pack_ins(uint32_t op, uint32_t dst, uint32_t src,
                                                uint32_t idx) {
  return op | (dst << 8) | (src << 16) | (idx << 24);
}

struct EpiProgram {
  int32_t n_ins;
  uint32_t ins[kMaxIns];
  float scalars[GE_MAX_SCALARS];
  int32_t n_tma_aux;                      // Load tensors, in first-use order
  int32_t tma_aux_slot[GE_MAX_TMA_AUX];   // their aux slots
  int32_t tma_aux_dtype[GE_MAX_TMA_AUX];
  int32_t n_bcast;                        // Broadcast vectors
  int32_t bcast_slot[GE_MAX_AUX];
  int32_t bcast_dtype[GE_MAX_AUX];
  int32_t n_cbcast;                       // column-broadcast vectors
  int32_t cbcast_slot[GE_MAX_AUX];
  int32_t cbcast_dtype[GE_MAX_AUX];
  int32_t n_out;
  int32_t out_dtype[GE_MAX_OUT];
  int32_t n_regs;                         // registers the program uses
};

// ---------------------------------------------------------------------------
// GEMM kernel parameter block (passed by value as a __grid_constant__).
// ---------------------------------------------------------------------------
constexpr int BM = 128;      // accumulator rows per CTA (TMEM lanes)
constexpr int BK = 64;       // 16-bit elements per k-block: one 128-byte swizzle row
constexpr int UMMA_K = 16;   // K of one tcgen05.mma.kind::f16
// Epilogue warps: one group of 4 (one warp per TMEM lane quarter) or two
// groups (8 warps, the groups taking alternate 32-column steps of the tile).
// A CTA has a producer warp, an MMA warp and an epilogue TMA warp ahead of
// the epilogue warps.
constexpr int kMaxEpiWarps = 8;
constexpr int kMaxEpiGroups = kMaxEpiWarps / 4;
constexpr int kEpiWarp0 = 3;   // first epilogue warp
constexpr int kEpiRows = 128;  // rows of a staged epilogue box: all of a CTA's accumulator rows
__host__ __device__ constexpr int threads_for(int epi_warps) { return 32 * kEpiWarp0 + 32 * epi_warps; }
// Output staging boxes per epilogue group: two (a step's outputs are written
// while the previous step's box is still being stored) with one group; one
// per group with two, where the other group keeps the stores flowing.
constexpr int kMaxOutBufs = 2;
__host__ __device__ constexpr int out_bufs_for(int epi_warps) { return epi_warps == 8 ? 1 : 2; }
constexpr int kMaxStages = 8;
constexpr int kMaxAuxStages = 8;

// One problem of a grouped GEMM, in device memory (a table uploaded per run).
// Its tiles are [tile_begin, tile_end) of the launch's tile sequence; within
// the problem they are ordered like the tiles of one batch of a batched GEMM.
// The tile -> (problem, m block, n block, k blocks) map itself is a separate
// table (KParams::tile_info), fixed when the plan is made.
struct alignas(128) GroupDesc {
  CUtensorMap tmA;                    // (K, M, 1)
  CUtensorMap tmB;                    // (N, K, 1)
  CUtensorMap tmAux[GE_MAX_TMA_AUX];  // (N, M, 1)
  CUtensorMap tmOut[GE_MAX_OUT];      // (N, M, 1)
  const void *bcast_ptr[GE_MAX_AUX];
  const void *cbcast_ptr[GE_MAX_AUX];
  int32_t M, N, num_m_blk, num_n_blk, num_kb, tile_begin, tile_end, problem;
};

struct KParams {
  CUtensorMap tmA;                    // (K, M, L) box (64, 128, 1), 128B swizzle
  CUtensorMap tmB;                    // (N, K, L) box (64, 64, 1), 128B swizzle
  CUtensorMap tmAux[GE_MAX_TMA_AUX];  // (N, M, L) box (EW, kEpiRows, 1)
  CUtensorMap tmOut[GE_MAX_OUT];      // (N, M, L) box (EW, kEpiRows, 1)
  const void *bcast_ptr[GE_MAX_AUX];
  const void *cbcast_ptr[GE_MAX_AUX];
  uint32_t *status;                   // device status word (timeouts)
  EpiProgram prog;
  int32_t L, M, N, K;
  int32_t ab_bf16;                     // A/B are bf16 (else fp16)
  int32_t num_m_blk, num_n_blk, num_tiles, num_kb;
  int32_t num_full;  // tiles [0, num_full) are full width; each later pair of
                     // tiles is the two column halves of one split tile
  int32_t raster_group;
  int32_t stages, aux_stages;
  uint32_t off_A, off_B, off_aux, off_out, off_bar;  // byte offsets in dynamic smem
  uint32_t aux_stage_bytes, out_stage_bytes;          // one staging slot: a kEpiRows x EW box
                                                      // per aux tensor / per output
  uint32_t aux_off[GE_MAX_TMA_AUX], out_off[GE_MAX_OUT];
  uint32_t tx_bytes;      // bytes one k-block stage receives (both CTAs of a pair)
  uint32_t tx_bytes_half; // the same for a half-width tile
  uint32_t aux_tx_bytes;  // bytes one aux staging slot receives
  uint32_t b_lbo, b_sbo;  // B smem descriptor strides (bytes)
  uint64_t timeout_ns;
  uint32_t debug_flags;
  int32_t a_mn;             // A stored M-major ((L,K,M), M contiguous), else K-major
  int32_t b_k;              // B stored K-major ((L,N,K), K contiguous), else N-major
  int32_t cd_m;             // epilogue tensors and outputs M-major ((L,N,M)), else N-major
  const GroupDesc *groups;  // grouped GEMM: the problem table (else nullptr)
  const int4 *tile_info;    // grouped GEMM: per tile {problem entry, m block, n block, k blocks}
  int32_t num_groups;
};

// Unfused elementwise kernel parameters.
struct EwParams {
  const float *acc;                   // (L, M, N) fp32 workspace
  const void *aux_ptr[GE_MAX_TMA_AUX];
  const void *bcast_ptr[GE_MAX_AUX];
  const void *cbcast_ptr[GE_MAX_AUX];
  void *out_ptr[GE_MAX_OUT];
  EpiProgram prog;
  int64_t rows;                       // L*M
  int32_t M;
  int32_t N;
  int32_t chunks_per_row;             // ceil(N / 8): one thread per 8 columns
  int32_t cd_m;                       // aux tensors and outputs M-major ((L,N,M))
};

// Where a device-side wait gave up (second word of the status block).
enum WaitSite : uint32_t {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_FULL = 2,
  SITE_MMA_TMEM_EMPTY = 3,
  SITE_EPI_TMEM_FULL = 4,
  SITE_EPI_AUX_FULL = 5,
  SITE_DRAIN = 6,
  SITE_EPI_TMA = 7,        // the epilogue TMA thread saw no progress
  SITE_EPI_OUT_EMPTY = 8,  // an epilogue warp waited for an output box
};

}  // namespace ge
