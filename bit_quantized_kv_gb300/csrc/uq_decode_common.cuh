// uq_decode_common.cuh -- definitions shared by the decode kernels: page
// geometry and the caller-owned workspace layout (split partials and the
// device-side plan).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "uq_device.cuh"

namespace uq {

// L2 sector promotion of the page copies (CUtensorMapL2promotion: 0 none,
// 1 64 B, 2 128 B, 3 256 B).
#ifndef UQ_KV_L2_PROMOTION
#define UQ_KV_L2_PROMOTION 1
#endif
constexpr int kPage = 16;                        // tokens per tile (the smallest block_size)
constexpr int kTileBytes = kPage * kSlotBytes;   // 4352 bytes per (tile, kv head)
#ifndef UQ_MIN_PAGES_PER_UNIT
#define UQ_MIN_PAGES_PER_UNIT 8
#endif
// Fixed cost of a work unit in tiles, per stage-1 instantiation: the 16-row
// kernel's unit start and merge cost more (16-row query prologue, tensor
// memory zeroing, two-part merge).
#ifndef UQ_UNIT_COST_TILES_8ROW
#define UQ_UNIT_COST_TILES_8ROW 48
#endif
#ifndef UQ_UNIT_COST_TILES_16ROW
#define UQ_UNIT_COST_TILES_16ROW 64
#endif
#ifndef UQ_S1_NSTAGE
#define UQ_S1_NSTAGE 2
#endif
#ifndef UQ_S1_MIN_BLOCKS
#define UQ_S1_MIN_BLOCKS 4
#endif
constexpr int kMinPagesPerUnit = UQ_MIN_PAGES_PER_UNIT;  // floor of 128 tokens per split
constexpr float kUnitCostTiles8 = UQ_UNIT_COST_TILES_8ROW;    // work units per CTA = sqrt(tiles / this)
constexpr float kUnitCostTiles16 = UQ_UNIT_COST_TILES_16ROW;
#ifndef UQ_MIN_UNITS_PER_CTA
#define UQ_MIN_UNITS_PER_CTA 2
#endif
#ifndef UQ_MAX_UNITS_PER_CTA
#define UQ_MAX_UNITS_PER_CTA 8
#endif
constexpr int kMinUnitsPerCta = UQ_MIN_UNITS_PER_CTA, kMaxUnitsPerCta = UQ_MAX_UNITS_PER_CTA;
constexpr int kStage1Stages = UQ_S1_NSTAGE;              // pages in flight per warp
// 16-row query groups keep O^T (128 fp32 per lane) in tensor memory: 128
// columns over all 128 lanes per CTA, each warp in its own 32 lanes.  That
// frees the registers for 3 resident CTAs per SM (4 would need <= 128).
constexpr uint32_t kTmemCols = 128;
#ifndef UQ_S1_NT2_MIN_BLOCKS
#define UQ_S1_NT2_MIN_BLOCKS 3
#endif
constexpr int kTmemCtasPerSm = UQ_S1_NT2_MIN_BLOCKS;
// The general 16-row instantiation (windows, larger pages, multi-query units)
// runs 4 CTAs per SM at 128 registers: measured 9.7% faster on a multi-query
// chunk, where the plain copy at 4 CTAs is 3.5% slower on a long batch.
#ifndef UQ_S1_NT2_GEN_MIN_BLOCKS
#define UQ_S1_NT2_GEN_MIN_BLOCKS 4
#endif
constexpr int kTmemCtasPerSmGen = UQ_S1_NT2_GEN_MIN_BLOCKS;
#ifndef UQ_PLAN_THREADS
#define UQ_PLAN_THREADS 256
#endif
constexpr int kPlanThreads = UQ_PLAN_THREADS;
constexpr float kLog2e = 1.4426950408889634f;
// A running softmax maximum (log2 units) moves only when a page's maximum
// exceeds it by more than this, so probabilities stay below 2^8.
constexpr float kLazyMaxLog2 = 8.f;

// ---------------------------------------------------------------------------
// Workspace layout (caller-owned, no initialisation needed).
// ---------------------------------------------------------------------------
struct Workspace {
  float* part_o;       // [B][Hq][S][256] split outputs, normalised
  float* part_lse;     // [B][Hq][S]      log2-sum-exp of each split
  uint32_t* units;     // [<= S * B * Hk] b | split << 16 | kv_head << 24
  int2* seq_info;      // [B] (pages per split, active splits)
  int* order;          // [B] sequences with at least one page, longest split first
  int* hdr;            // [0] number of units, [1] next unit to take, [2] units to redo
  uint32_t* redo;      // [<= S * B * Hk] units whose stage-1 result needs the exact pass
};

__host__ __device__ inline size_t workspace_bytes(int B, int Hq, int S) {
  const size_t rows = (size_t)B * Hq * S;
  const size_t bytes = rows * kHeadDim * 4 + rows * 4 + rows * 4 + (size_t)B * 8 +
                       (size_t)B * 4 + 64;
  return (bytes + 255) / 256 * 256;
}

__host__ __device__ inline Workspace workspace_layout(void* base, int B, int Hq, int S) {
  const size_t rows = (size_t)B * Hq * S;
  uint8_t* p = static_cast<uint8_t*>(base);
  Workspace w;
  w.part_o = reinterpret_cast<float*>(p);
  p += rows * kHeadDim * 4;
  w.part_lse = reinterpret_cast<float*>(p);
  p += rows * 4;
  w.units = reinterpret_cast<uint32_t*>(p);
  p += rows * 4;
  w.seq_info = reinterpret_cast<int2*>(p);   // rows * 1032 is a multiple of 8
  p += (size_t)B * 8;
  w.order = reinterpret_cast<int*>(p);
  p += (size_t)B * 4;
  w.hdr = reinterpret_cast<int*>(p);
  // at most S * B * Hk <= rows / 6 units (6 or more query heads per kv
  // head): the upper half of the units array holds the redo list
  w.redo = w.units + rows / 2;
  return w;
}

__device__ __forceinline__ int clamp_len(int L, int max_blocks) {
  L = max(L, 0);
  const long long cap = (long long)max_blocks * kPage;
  return (long long)L > cap ? (int)cap : L;
}

// Where the decode kernels find each row's length and pages.  A batch reads
// seq_lens[b] and block-table row b (bt_stride = the table's width).  A
// multi-query chunk (mq_base >= 0) gives row b the length mq_base + b + 1
// and every row the same pages (bt_stride = 0), as the synthetic lengths
// arange(cached + 1, L + 1) and expanded block table of a continuation chunk.
// A sliding window (window > 0) keeps the last `window` tokens of each row.
// The kernels walk rows in 16-token tiles; a cache page of block_size tokens
// holds 2^lg_tpp tiles, and a row can hold at most cap_tiles tiles (the
// block-table width times the tiles per page).
struct SeqRows {
  const int32_t* seq_lens;
  int64_t bt_stride;
  int mq_base;
  int window;
  int lg_tpp;
  int cap_tiles;
  int pack;    // rows (sequences or chunk positions) per work unit: 1, or 2 for multi-query
  int n_rows;  // rows in the call (B, or the chunk length)
};

__device__ __forceinline__ int row_len(const SeqRows& r, int b) {
  return clamp_len(r.mq_base >= 0 ? r.mq_base + b + 1 : r.seq_lens[b], r.cap_tiles);
}

// First token a row of length L attends to.
__device__ __forceinline__ int row_lo(const SeqRows& r, int L) {
  return (r.window > 0 && L > r.window) ? L - r.window : 0;
}

// A unit row u covers rows u*pack .. u*pack+pack-1 (those < n_rows).  With
// pack > 1 the rows are chunk positions, whose lengths grow by one per
// position, so the unit reads from the first row's window start to the last
// row's length.
__device__ __forceinline__ int unit_last_row(const SeqRows& r, int u) {
  return min(u * r.pack + r.pack - 1, r.n_rows - 1);
}
__device__ __forceinline__ int unit_len(const SeqRows& r, int u) { return row_len(r, unit_last_row(r, u)); }
__device__ __forceinline__ int unit_lo(const SeqRows& r, int u) { return row_lo(r, row_len(r, u * r.pack)); }
__device__ __forceinline__ int unit_pages(const SeqRows& r, int u) {
  return (unit_len(r, u) + kPage - 1) / kPage - unit_lo(r, u) / kPage;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

}  // namespace uq
