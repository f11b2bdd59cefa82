// uq_decode.cu -- split-KV paged decode attention over the FP4 E2M1 + UE8M0
// cache (vllm.v1.attention.ops.flydsl_ultraquant_decode,
// flydsl_ultraquant_decode_attention: query prologue with the E4M3 haircut,
// stage-1 split partials, partition reduce; the fixed split count follows
// vllm.v1.attention.ops.turboquant_soa.triton_turboquant_decode_v2).
//
// Three kernels on the caller's stream:
//
// Plan (one CTA).  Reads seq_lens and chooses, for the whole batch, one unit
// size T (pages of one kv head) so that the batch splits into U work units
// per resident stage-1 CTA, never below kMinPagesPerUnit pages.  Each unit
// costs a fixed start (first copies in flight, query prologue, merge and
// partial write) while the last units decide the tail, which grows with
// the unit size; the sum is smallest near U = sqrt(work per CTA / 2 fixed
// cost), which with the measured costs is U = sqrt(tiles per CTA / c),
// kept in [2, 8], with c = 48 tiles for 6- and 8-row query groups and 64
// for 16-row ones.  Sequence b gets n_b = min(S, ceil(P_b / T)) splits
// of whole pages.  Units (sequence, split, kv head) are listed with the
// longest units first; the plan also resets the unit counter.  For a
// multi-query chunk the "sequences" are unit rows of one or two chunk
// positions (SeqRows::pack) that read the same pages; with equal split
// counts their units are listed split-major so that units reading the same
// pages run side by side.
//
// Stage 1 (persistent: resident CTAs only, 4 warps each).  Each CTA takes
// units from the counter.  Inside a unit each warp takes every 4th page and
// keeps its own online-softmax state; a page's 16 slots of one kv head
// (16 x 272 B, strided by Hk * 272 B in the cache) arrive in shared memory as
// one TMA tile copy (a 3-D tensor map over the cache: 68 words x Hk heads x
// slots, box 68 x 1 x 16) completing on a per-stage mbarrier, NSTAGE pages
// ahead.  One lane issues each copy with warp-uniform operands.  The unit's
// query rows (6, 8 or 16, or two chunk positions of 6 or 8) are rotated
// (fp32 butterfly, x 1/16), rounded through E4M3 and kept in shared memory
// as f16 in tensor-core operand order.  At the end of the unit the four
// warps' states are merged into one split partial.
//
// Tensor-core formulation (mma.m16n8k16, f16 in, fp32 accumulate):
//   QK:  S[t, r] = sum_d K'[t, d] Q'[r, d]      (M = 16 tokens, N = 8 rows)
//   PV:  O^T[d, r] += sum_t V'[t, d] W[r, t]    (M = 16 head dims, N = 8 rows)
// Every FP4 value is c * 2^(e_blk - 127).  For each token t the largest
// block exponent E_t is factored out: K' = c * 2^(13 + e_blk - E_t) and
// V' = c * 2^(13 + e_blk - E_t) are exact f16 values for e_blk > E_t - 28
// (every kept factor is a normal f16, the largest code 6 * 2^13 stays inside
// f16's range).  2^(E^K_t - 127 - 13) multiplies the scores;
// E^V_t - 127 - 13 is added to the exponent of the probability that weights
// the token's V' row.  A K block 2^28 or more below its token's largest
// block turns that token's score factor NaN, and the unit is redone in
// plain fp32 by the exact pass; a V block that far below its token's
// largest block is dropped (its share of an output is below 2^-28 of that
// token's).  The contraction index of QK may be permuted freely as
// long as Q' and K' agree, which lets every lane read contiguous bytes:
// lane (g = lane/4, c = lane%4) owns head dims [64c, 64c+64) of K (k-step i
// covers 64c + 4i .. +3) and V head dims [32g, 32g+32) (one UE8M0 block).
//
// 16-row query groups keep O^T in tensor memory instead of registers: 128
// fp32 per lane would hold a thread above 168 registers and the SM at 8
// warps.  Each CTA allocates 128 TMEM columns over its 128 lanes; warp w
// works in lanes 32w .. 32w+31 only, as per-thread storage.  PV brings in
// the O^T columns of one V word in two 16-column halves, each loaded while
// the previous half's MMAs run, and stores them back; the rare rescale and
// the final merge go through the same columns.  Three CTAs (12 warps) fit
// per SM.
//
// Stage 2: one warp per (sequence, query head) merges the active splits with
// the log-sum-exp rule and writes bf16.
//
// Stage 1 and stage 2 are launched with programmatic stream serialization:
// each may start its set-up while the kernel before it finishes, and waits
// in griddepcontrol.wait before reading that kernel's output.
#include <mutex>
#include <type_traits>

#include <cuda_fp16.h>

#include "uq_decode_common.cuh"

namespace uq {

// ---------------------------------------------------------------------------
// Plan.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads)
decode_plan(const SeqRows rows, int B, int Hk, int S,
            int grid, float unit_cost_tiles, Workspace ws) {
  __shared__ long long s_part[kPlanThreads / 32];
  __shared__ int s_hist[32], s_cursor[32], s_wsum[kPlanThreads / 32];
  __shared__ long long s_total;
  __shared__ int s_nseq, s_nact_min, s_nact_max;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The plan is queued with programmatic serialization, so its launch
  // overlaps the kernel before it on the stream; everything it reads or
  // writes waits for that kernel to finish.
  pdl_wait();
  pdl_launch_dependents();   // stage 1 may start its set-up now
  if (tid < 32) s_hist[tid] = 0;
  if (tid == 0) {
    s_nact_min = 1 << 30;
    s_nact_max = 0;
  }

  long long mine = 0;
  for (int b = tid; b < B; b += kPlanThreads) mine += unit_pages(rows, b);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, m);
  if (lane == 0) s_part[warp] = mine;
  __syncthreads();
  if (tid == 0) {
    long long t = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) t += s_part[w];
    s_total = t;
  }
  __syncthreads();
  const long long work = s_total * Hk;
  const float per_cta = (float)work / (float)max(grid, 1);
  const int upc = min(kMaxUnitsPerCta, max(kMinUnitsPerCta, (int)sqrtf(per_cta / unit_cost_tiles)));
  const long long target_units = (long long)grid * upc;
  long long T = (work + target_units - 1) / target_units;
  if (T < kMinPagesPerUnit) T = kMinPagesPerUnit;

  for (int b = tid; b < B; b += kPlanThreads) {
    const int P = unit_pages(rows, b);
    int n = 0, pps = 0, nact = 0;
    if (P > 0) {
      const long long want = (P + T - 1) / T;
      n = (int)(want < S ? want : S);
      n = max(n, 1);
      pps = (P + n - 1) / n;
      nact = (P + pps - 1) / pps;
      atomicAdd(&s_hist[31 - __clz(pps)], 1);
    }
    ws.seq_info[b] = make_int2(pps, nact);
    atomicMin(&s_nact_min, nact);
    atomicMax(&s_nact_max, nact);
  }
  __syncthreads();
  if (rows.mq_base >= 0 && s_nact_min == s_nact_max && s_nact_max > 0) {
    // Multi-query unit rows read the same pages.  With equal split counts the
    // units are listed split-major, (split, kv head, unit row), so the units
    // that read the same pages run side by side and the repeats hit L2.
    const int per_split = Hk * B, total = s_nact_max * per_split;
    for (int idx = tid; idx < total; idx += kPlanThreads) {
      const int s = idx / per_split, rem = idx - s * per_split, g = rem / B, b = rem - g * B;
      ws.units[idx] = (uint32_t)b | ((uint32_t)s << 16) | ((uint32_t)g << 24);
    }
    if (tid == 0) {
      ws.hdr[0] = total;
      ws.hdr[1] = grid;   // units 0 .. grid-1 are each CTA's first
      ws.hdr[2] = 0;
    }
    return;
  }
  if (tid == 0) {
    int acc = 0;
    for (int k = 31; k >= 0; --k) {   // longest splits first
      s_cursor[k] = acc;
      acc += s_hist[k];
    }
    s_nseq = acc;
  }
  __syncthreads();
  for (int b = tid; b < B; b += kPlanThreads) {
    const int pps = ws.seq_info[b].x;
    if (pps > 0) ws.order[atomicAdd(&s_cursor[31 - __clz(pps)], 1)] = b;
  }
  __syncthreads();

  // units: exclusive prefix over the ordered sequences of (active splits * Hk)
  const int nseq = s_nseq;
  const int chunk = (nseq + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(nseq, tid * chunk), hi = min(nseq, lo + chunk);
  int cnt = 0;
  for (int k = lo; k < hi; ++k) cnt += ws.seq_info[ws.order[k]].y * Hk;
  int incl = cnt;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, m);
    if (lane >= m) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
      const int t = s_wsum[w];
      s_wsum[w] = acc;
      acc += t;
    }
  }
  __syncthreads();
  int off = s_wsum[warp] + incl - cnt;
  for (int k = lo; k < hi; ++k) {
    const int b = ws.order[k];
    const int nact = ws.seq_info[b].y;
    for (int s = 0; s < nact; ++s)
      for (int g = 0; g < Hk; ++g) ws.units[off++] = (uint32_t)b | ((uint32_t)s << 16) | ((uint32_t)g << 24);
  }
  if (tid == kPlanThreads - 1) {
    ws.hdr[0] = off;   // the last thread's range ends the list
    ws.hdr[1] = grid;  // units 0 .. grid-1 are each CTA's first
    ws.hdr[2] = 0;
  }
}

// ---------------------------------------------------------------------------
// Stage 1.
// ---------------------------------------------------------------------------
// q' = f16(e4m3(q H / 16)) for one query row (bf16, 256 head dims) by one
// warp: lane loads head dims 8*lane .. 8*lane+7, the Walsh-Hadamard butterflies
// run in registers (strides 1..4) and across lanes (strides 8..128), and the
// lane returns its 8 dims as four f16x2 (the lower dim in the low half).
__device__ __forceinline__ void query_prime8(const uint16_t* __restrict__ q_row, int lane, uint32_t (&pk)[4]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(q_row + lane * 8);
  float x[8];
  const uint32_t uu[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_bits_to_f32(uu[i] & 0xffffu);
    x[2 * i + 1] = bf16_bits_to_f32(uu[i] >> 16);
  }
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & h) == 0) {
        const float a = x[i], cc = x[i + h];
        x[i] = a + cc;
        x[i + h] = a - cc;
      }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float sgn = (lane & m) ? -1.f : 1.f;   // upper lane: other - own
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = fmaf(x[i], sgn, other);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) pk[i] = e4m3_roundtrip_f16x2(x[2 * i] * 0.0625f, x[2 * i + 1] * 0.0625f);
}

// 2^e as fp32 for an integer e <= 0 (subnormal below -126, 0 below -149).
__device__ __forceinline__ float pow2_nonpos(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23)
                   : (e >= -149 ? __uint_as_float(1u << (e + 149)) : 0.f);
}

// The exact pass over the pages of a work unit, for units that hold a token
// whose K blocks span 2^28 or more: the tensor-core pass keeps K block scales
// relative to the token's largest block as f16 and cannot hold such a block
// exactly.  Such spreads do not come out of a rotated K in practice; the pass
// exists so that scores stay exact for every cache the store can write.
// Everything here is plain fp32 on the CUDA cores, read straight from the
// cache in global memory: score s = scale*log2e * sum over blocks of
// 2^(byte - 127) * (E2M1 codes . q'), then the same online softmax state as
// the main loop -- m (running maximum), d (V reference relative to m), l (sum
// of 2^(s - m)) -- with every update taken eagerly, and O accumulated with V
// taken relative to its token's largest block (2^(byte - E_V)) and weight
// 2^(s - m + E_V - 127 - d).
// Lane (gq, c) computes K block gq's share of every score of rows
// nt*8 + 2c + h (the 8 lanes of a row sum their shares), and accumulates O
// for head dims 32gq .. 32gq+31 of those rows: acc[mt][k] holds row
// nt*8 + 2c + (k & 1), head dim 32gq + 2mt + (k >> 1), the layout of the
// stage-1 kernel's O fragments.  q_rows points at row nt*8 + 2c of q' (f16,
// head dims in order, row stride q_row_bytes).  Returns the state of rows
// nt*8 + 2c + h in m, d, l (l whole in lane gq == 0, 0 elsewhere, so that
// the sum over the row's lanes is the row sum) and acc.
template <bool GEN>
__device__ __forceinline__ void exact_rows(const uint8_t* __restrict__ kv, const int32_t* __restrict__ bt_row,
                                           int num_blocks, int Hk, int g, int lg_tpp, int page0, int n_my,
                                           int page_step, int L, const int (&lo)[2], const int (&hi)[2],
                                           const uint8_t* q_rows, int q_row_bytes, float scale_log2e, int gq,
                                           float (&m)[2], float (&d)[2], float (&l)[2], float (&acc)[16][4]) {
  const int tile_mask = (1 << lg_tpp) - 1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    m[h] = -INFINITY;
    d[h] = -INFINITY;
    l[h] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  const int64_t tok_stride = (int64_t)Hk * kSlotBytes;
#pragma unroll 1
  for (int j = 0; j < n_my; ++j) {
    const int page = page0 + j * page_step;
    const int pid = bt_row[page >> lg_tpp];
    if ((unsigned)pid >= (unsigned)num_blocks) continue;   // reported by the main loop
    const int nval = min(kPage, L - page * kPage);
    const uint8_t* tile = kv + ((int64_t)((pid << lg_tpp) + (page & tile_mask)) * kPage * Hk + g) * kSlotBytes;
#pragma unroll 1
    for (int t = 0; t < nval; ++t) {
      const uint8_t* slot = tile + t * tok_stride;
      const uint4 kc = *reinterpret_cast<const uint4*>(slot + 16 * gq);
      const float kscale = scale_log2e * ue8m0_to_f32(slot[kKScaleOff + gq]);
      const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w};
      float part[2] = {0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t f[4];
        f16x2x4_from_e2m1_word(kw[w], f);
#pragma unroll
        for (int e8 = 0; e8 < 8; ++e8) {
          const float kval = __half2float(__ushort_as_half((unsigned short)(f[e8 >> 1] >> (16 * (e8 & 1)))));
          const int dim = 32 * gq + 8 * w + e8;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint16_t qb = *reinterpret_cast<const uint16_t*>(q_rows + h * q_row_bytes + 2 * dim);
            part[h] = fmaf(kval, __half2float(__ushort_as_half(qb)), part[h]);
          }
        }
      }
      float sc[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x = part[h] * kscale;
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) x += __shfl_xor_sync(0xffffffffu, x, msk);
        sc[h] = x;
      }
      const uint2 vs = *reinterpret_cast<const uint2*>(slot + kVScaleOff);
      const uint32_t Ev = max_byte8(vs.x, vs.y);
      const uint32_t vb = ((gq < 4 ? vs.x : vs.y) >> (8 * (gq & 3))) & 0xffu;
      const float vrel = pow2_nonpos((int)vb - (int)Ev);
      const float ev = (float)((int)Ev - 127);
      const uint4 vc = *reinterpret_cast<const uint4*>(slot + kVCodeOff + 16 * gq);
      const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
      const int tok = page * kPage + t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (GEN && (tok < lo[h] || tok >= hi[h])) continue;
        const float sv = sc[h];
        if (sv > m[h]) {
          if (m[h] != -INFINITY) {
            l[h] *= exp2f(m[h] - sv);
            d[h] += m[h] - sv;
          }
          m[h] = sv;
        }
        const float u = (sv - m[h]) + ev;
        if (u > d[h]) {
          if (d[h] != -INFINITY) {
            const float a = exp2f(d[h] - u);
#pragma unroll
            for (int mt = 0; mt < 16; ++mt) {
              acc[mt][h] *= a;
              acc[mt][2 + h] *= a;
            }
          }
          d[h] = u;
        }
        l[h] += exp2f(sv - m[h]);
        const float wt = exp2f(u - d[h]) * vrel;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t f[4];
          f16x2x4_from_e2m1_word(vw[w], f);
#pragma unroll
          for (int e8 = 0; e8 < 8; ++e8) {
            const float vval = __half2float(__ushort_as_half((unsigned short)(f[e8 >> 1] >> (16 * (e8 & 1)))));
            acc[4 * w + (e8 >> 1)][2 * (e8 & 1) + h] = fmaf(wt, vval, acc[4 * w + (e8 >> 1)][2 * (e8 & 1) + h]);
          }
        }
      }
    }
  }
  if (gq != 0) l[0] = l[1] = 0.f;
}

template <int NT, int NWARPS, int NSTAGE>
struct Stage1Layout {
  static constexpr int kRows = NT * 8;                       // padded query rows
  // 16-row groups keep O^T in tensor memory between pages (see kTmemCols)
  static constexpr bool kTmemO = NT == 2;
  static constexpr int kStageBytes = NWARPS * NSTAGE * kTileBytes;
  static constexpr int kMergeParts = kTmemO ? 2 : 1;         // head-dim parts merged in turn
  static constexpr int kPartDims = kHeadDim / kMergeParts;
  static constexpr int kORowStride = kPartDims + 4;          // floats
  static constexpr int kMergeBytes = NWARPS * kRows * kORowStride * 4;
  static constexpr int kUnionBytes = kStageBytes > kMergeBytes ? kStageBytes : kMergeBytes;
  static constexpr int kStatsOff = kUnionBytes;              // [NWARPS][kRows][4] floats
  static constexpr int kStatsBytes = NWARPS * kRows * 4 * 4;
  static constexpr int kRowInfoOff = kStatsOff + kStatsBytes; // [kRows][NWARPS+2] floats
  static constexpr int kRowInfoBytes = kRows * (NWARPS + 2) * 4;
  // per warp, per tile: [K, V][token] 8 relative block scales (f16) and one factor
  static constexpr int kMetaRelBytes = 2 * kPage * 16;
  static constexpr int kMetaWarpBytes = kMetaRelBytes + 2 * kPage * 4;
  static constexpr int kMetaOff = (kRowInfoOff + kRowInfoBytes + 15) / 16 * 16;
  static constexpr int kBarOff = kMetaOff + NWARPS * kMetaWarpBytes;
  static constexpr int kBarBytes = NWARPS * NSTAGE * 8;
  // unit id, abort flag, TMEM base, redo flag, (unused), next unit, its
  // work-list word
  static constexpr int kMiscOff = kBarOff + kBarBytes;
  static constexpr int kQOff = (kMiscOff + 32 + 127) / 128 * 128;
  static constexpr int kQRowBytes = kHeadDim * 2 + 16;       // padded: conflict-free ldmatrix
  static constexpr int kQBytes = kRows * kQRowBytes;
  static constexpr int kBytes = kQOff + kQBytes;
};

// GEN: 0 plain (block_size 16, no window, one query row per sequence);
// 1 multi-query unit rows only (rows of their own lengths; block_size 16,
// no window), which folds the window start and the page-size shifts away;
// 2 general (a sliding window or pages of more than 16 tokens as well).
template <int NT, int NWARPS, int NSTAGE, int GEN>
__global__ void __launch_bounds__(NWARPS * 32, NT == 1 ? UQ_S1_MIN_BLOCKS : (GEN ? kTmemCtasPerSmGen : kTmemCtasPerSm))
decode_stage1(const uint16_t* __restrict__ query, int64_t q_ss, int64_t q_sh,
              const __grid_constant__ CUtensorMap kv_map, const uint8_t* __restrict__ kv,
              const int32_t* __restrict__ block_table, const SeqRows rows, float scale_log2e, int Hq, int Hk,
              int QG, int num_blocks, int S, Workspace ws,
              unsigned* __restrict__ err) {
  using Lay = Stage1Layout<NT, NWARPS, NSTAGE>;
  constexpr int NCH = NT == 1 ? 4 : 2;   // independent QK accumulator chains per n-tile
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + Lay::kBarOff + warp * NSTAGE * 8;
  const uint32_t stage_base = smem_base + warp * NSTAGE * kTileBytes;
  const uint32_t meta_rel = smem_base + Lay::kMetaOff + warp * Lay::kMetaWarpBytes;
  const uint32_t meta_f = meta_rel + Lay::kMetaRelBytes;
  volatile int* s_misc = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff);
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + Lay::kQOff);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NWARPS * NSTAGE; ++i) mbar_init(smem_base + Lay::kBarOff + 8 * i, 1);
    s_misc[1] = 0;
    s_misc[3] = 0;
    fence_barrier_init();
  }
  if constexpr (Lay::kTmemO) {
    if (warp == 0) tmem_alloc(smem_base + Lay::kMiscOff + 8, kTmemCols);
    tc_fence_before_sync();
  }
  __syncthreads();
  // this warp's O^T columns: its own 32 lanes, columns 32q + 16nt + 4e + k hold
  // o[nt][4q + e][k]
  uint32_t o_taddr = 0;
  if constexpr (Lay::kTmemO) {
    tc_fence_after_sync();
    o_taddr = (uint32_t)s_misc[2] + ((uint32_t)(32 * warp) << 16);
  }

  pdl_launch_dependents();   // stage 2 may be scheduled as CTAs retire
  pdl_wait();                // the plan's work list is complete
  const int n_units = ws.hdr[0];
  uint32_t tiles_done = 0;   // this warp's tiles so far: drives stage and parity
  uint32_t stage_ok = 0;     // bit s: stage s holds a page that was really copied
  const int ta = 2 * c, tb = 2 * c + 1, tcc = 2 * c + 8, td = 2 * c + 9;

  // The next unit and its work-list word (s_misc[5], s_misc[6]): a CTA's
  // first unit is its own index (the plan starts the counter at the grid
  // size); later ones are taken from the counter during the previous unit's
  // merge, so that the next unit's copies go out without waiting on it.
  if (threadIdx.x == 0) {
    s_misc[5] = (int)blockIdx.x;
    s_misc[6] = (int)blockIdx.x < n_units ? (int)ws.units[blockIdx.x] : 0;
  }

  for (;;) {
    if (threadIdx.x == 0) s_misc[0] = s_misc[1] ? n_units : s_misc[5];
    __syncthreads();
    const int u = s_misc[0];
    if (u >= n_units || s_misc[1]) break;
    const uint32_t unit = (uint32_t)s_misc[6];
    const int b = (int)(unit & 0xffffu), split = (int)((unit >> 16) & 0xffu), g = (int)(unit >> 24);
    const int L = GEN ? unit_len(rows, b) : row_len(rows, b);
    const int pps = ws.seq_info[b].x;
    const int P = (L + kPage - 1) / kPage;
    const int lo = GEN == 2 ? unit_lo(rows, b) : 0;   // first token of the window
    // Query rows of the unit: row r is query head g*QG + r % QG of row
    // b*pack + r / QG (pack > 1 only for multi-query chunk positions).
    const int pack = GEN ? rows.pack : 1;
    const int last_row = GEN ? unit_last_row(rows, b) : b;
    auto row_of = [&](int r) { return GEN ? min(b * pack + r / QG, last_row) : b; };
    auto row_exists = [&](int r) { return GEN ? r < QG * pack && b * pack + r / QG <= last_row : r < QG; };
    auto head_of = [&](int r) { return g * QG + (GEN ? r % QG : r); };
    // this lane's score rows nt*8 + 2c + h: their own token range [rlo, rhi)
    int rlo[NT][2], rhi[NT][2];
    if constexpr (GEN) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          rhi[nt][h] = row_len(rows, row_of(nt * 8 + 2 * c + h));
          rlo[nt][h] = GEN == 2 ? row_lo(rows, rhi[nt][h]) : 0;
        }
    }
    const int lg_tpp = GEN == 2 ? rows.lg_tpp : 0;
    const int p_begin = lo / kPage + split * pps;
    const int p_end = min(p_begin + pps, P);

    // ---- per-warp page schedule ---------------------------------------------
    const int n_pages = p_end - p_begin;
    const int n_my = n_pages > warp ? (n_pages - warp + NWARPS - 1) / NWARPS : 0;
    // tile t of the row is tile t % 2^lg_tpp of page block_table[b][t >> lg_tpp]
    const int32_t* bt_row = block_table + (int64_t)b * rows.bt_stride;
    const int tile_mask = (1 << lg_tpp) - 1;
    int pid_chunk = -1, pid_reg = -1;

    auto issue = [&](int j, int stg) {
      const int chunk = j >> 5;
      const int tile = p_begin + warp + j * NWARPS;
      if (chunk != pid_chunk) {
        const int jj = chunk * 32 + lane;
        pid_reg = jj < n_my ? bt_row[(p_begin + warp + jj * NWARPS) >> lg_tpp] : -1;
        pid_chunk = chunk;
      }
      const int pid = __shfl_sync(0xffffffffu, pid_reg, j & 31);
      const uint32_t bar = bar_base + 8 * stg;
      const bool ok = (unsigned)pid < (unsigned)num_blocks;
      stage_ok = ok ? (stage_ok | (1u << stg)) : (stage_ok & ~(1u << stg));
#ifdef UQ_TEST_STUCK_TILE
      // Test builds only: the first tile of work unit 0's first warp is
      // announced to its barrier but never copied, so that barrier's phase
      // cannot complete and the bounded wait on it runs out.  No copy is in
      // flight for that stage.
      const bool copy = !(u == 0 && warp == 0 && j == 0);
#else
      constexpr bool copy = true;
#endif
      // the warp has finished reading this stage (callers __syncwarp first)
      if (lane == 0) {
        if (ok) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(bar, kTileBytes);
          if (copy)
            tma_load_3d(stage_base + stg * kTileBytes, &kv_map, 0, g,
                        ((pid << lg_tpp) + (tile & tile_mask)) * kPage, bar);
        } else {
          atomicOr(err, kErrBadPage);
          mbar_arrive(bar);
        }
      }
    };

    // this unit's first tile lands in stage tiles_done % NSTAGE, phase parity
    // (tiles_done / NSTAGE) & 1; later tiles advance both incrementally
    const int stg0 = (int)(tiles_done % NSTAGE);
    const uint32_t ph0 = (tiles_done / NSTAGE) & 1u;
    for (int j = 0; j < NSTAGE && j < n_my; ++j) issue(j, (stg0 + j) % NSTAGE);

    // ---- query prologue: q' = f16(e4m3(fp32(q) H)) in operand order -----------
    // Row r, k-step i, position kp holds head dim 64c + 4i + e with
    // kp = 2c + (e & 1) + 8 (e >> 1).
    for (int r = warp; r < Lay::kRows; r += NWARPS) {
      uint8_t* row = reinterpret_cast<uint8_t*>(qs) + r * Lay::kQRowBytes;
      uint32_t pk[4] = {0u, 0u, 0u, 0u};
      if (row_exists(r))
        query_prime8(query + (int64_t)row_of(r) * q_ss + (int64_t)head_of(r) * q_sh, lane, pk);
      // lane holds head dims 8*lane .. 8*lane+7: c' = lane / 8, k-steps 2(lane % 8) + {0, 1}
      const int cq = lane >> 3, i0 = 2 * (lane & 7);
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        uint8_t* kstep = row + (i0 + ii) * 32;
        *reinterpret_cast<uint32_t*>(kstep + 4 * cq) = pk[2 * ii];          // kp 2c', 2c'+1
        *reinterpret_cast<uint32_t*>(kstep + 16 + 4 * cq) = pk[2 * ii + 1]; // kp 2c'+8, 2c'+9
      }
    }
    __syncthreads();

    // ldmatrix row addresses: lane -> matrix lane/8 (k-step +(lane>>4), half (lane>>3)&1), row lane%8
    const uint32_t q_lds = smem_u32(qs) + (lane & 7) * Lay::kQRowBytes + (lane >> 4) * 32 + ((lane >> 3) & 1) * 16;

    // ---- main loop over this warp's pages -------------------------------------
    float o[NT][16][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int mt = 0; mt < 16; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    if constexpr (Lay::kTmemO) {
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_st32(o_taddr + 32 * q, z);
    }
    // Per score row: m_run the running score maximum (log2 units), d_run the
    // V reference relative to it (the probability that weights a token's V'
    // row is 2^(s - m_run + e_V - d_run)), l_run the sum of 2^(s - m_run).
    // Keeping the V reference relative to m_run keeps every exponent small
    // even when the scores themselves are large.
    float m_run[NT][2], d_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        m_run[nt][h] = -INFINITY;
        d_run[nt][h] = -INFINITY;
        l_run[nt][h] = 0.f;
      }

    bool timed_out = false;
    int j = 0;
    int stg = stg0;
    uint32_t phase = ph0;
    for (; j < n_my; ++j) {
      // With O^T in tensor memory the warp gives up together, so its
      // warp-collective tcgen05 instructions always run converged.
      bool arrived = mbar_wait(bar_base + 8 * stg, phase);
      if constexpr (Lay::kTmemO) arrived = __all_sync(0xffffffffu, arrived);
      if (!arrived) {
        timed_out = true;
        break;
      }
      const int page = p_begin + warp + j * NWARPS;
      const int nvalid = ((stage_ok >> stg) & 1u) ? min(kPage, L - page * kPage) : 0;
      if (nvalid > 0) {
        const uint32_t sb = stage_base + stg * kTileBytes;
        // -- tile metadata, one (token, K or V) scale row per lane: the token's
        //    largest block byte E, the 8 relative scales 2^(13 + byte - E) as
        //    f16 and one fp32 factor (K: scale*log2e*2^(E-127-13); V:
        //    E-127-13).  A token with a K block 2^28 or more below its
        //    largest block gets a NaN K factor instead: its scores, and so
        //    this lane's running sum, turn NaN, and the merge below hands
        //    the unit to the exact pass (rare).
        {
          const int mtok = lane & 15, kind = lane >> 4;
          const uint2 sc = lds64(sb + mtok * kSlotBytes + kKScaleOff + 8 * kind);
          const uint32_t E = max_byte8(sc.x, sc.y);
          // d = E - byte for all four bytes of a word at once (E is the
          // largest byte, so no byte borrows), then two per word spread to
          // halfwords and turned into f16 powers of two
          const uint32_t E4 = E * 0x01010101u;
          const uint32_t dx = E4 - sc.x, dy = E4 - sc.y;
          uint32_t p[4];
          p[0] = pow2_rel_f16x2(__byte_perm(dx, 0, 0x4140));
          p[1] = pow2_rel_f16x2(__byte_perm(dx, 0, 0x4342));
          p[2] = pow2_rel_f16x2(__byte_perm(dy, 0, 0x4140));
          p[3] = pow2_rel_f16x2(__byte_perm(dy, 0, 0x4342));
          sts128(meta_rel + (kind * kPage + mtok) * 16, make_uint4(p[0], p[1], p[2], p[3]));
          const float f = kind != 0 ? (float)((int)E - 127 - kRelTop)
                        : (any_rel_zero(p[0], p[1], p[2], p[3]) ? __uint_as_float(0x7fc00000u)
                                                                 : scale_log2e * ue8m0_rel_to_f32(E));
          sts32(meta_f + (kind * kPage + mtok) * 4, __float_as_uint(f));
        }
        __syncwarp();
        // K relative scales of tokens gq, gq+8 for blocks 2c, 2c+1 as f16x2 (both halves)
        const uint32_t kr0 = lds32(meta_rel + gq * 16 + 4 * c);
        const uint32_t kr1 = lds32(meta_rel + (gq + 8) * 16 + 4 * c);
        const uint32_t rk0[2] = {__byte_perm(kr0, 0, 0x1010), __byte_perm(kr0, 0, 0x3232)};
        const uint32_t rk1[2] = {__byte_perm(kr1, 0, 0x1010), __byte_perm(kr1, 0, 0x3232)};
        // -- QK on the tensor cores, NCH independent accumulation chains
        const uint4 ka0 = lds128(sb + gq * kSlotBytes + 32 * c);
        const uint4 ka1 = lds128(sb + gq * kSlotBytes + 32 * c + 16);
        const uint4 kb0 = lds128(sb + (gq + 8) * kSlotBytes + 32 * c);
        const uint4 kb1 = lds128(sb + (gq + 8) * kSlotBytes + 32 * c + 16);
        const uint32_t kaw[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t kbw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
        float sacc[NT][NCH][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) sacc[nt][ch][0] = sacc[nt][ch][1] = sacc[nt][ch][2] = sacc[nt][ch][3] = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t fa[4], fb[4];
          f16x2x4_from_e2m1_word(kaw[q], fa);
          f16x2x4_from_e2m1_word(kbw[q], fb);
          const uint32_t ra = rk0[q >> 2], rb = rk1[q >> 2];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            fa[e] = hmul2(fa[e], ra);
            fb[e] = hmul2(fb[e], rb);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t b0, b1, b2, b3;   // k-step 2q: (b0, b1), k-step 2q+1: (b2, b3)
            ldmatrix_x4(q_lds + nt * 8 * Lay::kQRowBytes + q * 64, b0, b1, b2, b3);
            mma_f16_16816(sacc[nt][(2 * q) % NCH], fa[0], fb[0], fa[1], fb[1], b0, b1);
            mma_f16_16816(sacc[nt][(2 * q + 1) % NCH], fa[2], fb[2], fa[3], fb[3], b2, b3);
          }
        }
        // -- V relative scales of tokens 2c, 2c+1, 2c+8, 2c+9 for block gq, and the
        //    K / V factors of tokens gq, gq+8
        const uint32_t vrel = meta_rel + kPage * 16 + 2 * gq;
        const uint32_t rv01 = __byte_perm(lds16(vrel + ta * 16), lds16(vrel + tb * 16), 0x5410);
        const uint32_t rv89 = __byte_perm(lds16(vrel + tcc * 16), lds16(vrel + td * 16), 0x5410);
        const float fk0 = __uint_as_float(lds32(meta_f + gq * 4));
        const float fk1 = __uint_as_float(lds32(meta_f + (gq + 8) * 4));
        const float evf0 = __uint_as_float(lds32(meta_f + (kPage + gq) * 4));
        const float evf1 = __uint_as_float(lds32(meta_f + (kPage + gq + 8) * 4));

        // -- scores and online softmax.  Both running maxima move lazily: only
        //    when a page's maximum exceeds the reference by more than
        //    kLazyMaxLog2, so a probability stays below 2^kLazyMaxLog2 (f16 keeps
        //    its full relative precision there) and rescaling O is rare.
        // tokens gq and gq + 8 of this page: valid for every score row (plain),
        // or against each row's own range [rlo, rhi) (GEN)
        const bool v0 = gq < nvalid, v1 = gq + 8 < nvalid;
        bool v0r[NT][2], v1r[NT][2];
        if constexpr (GEN) {
          const int t0 = page * kPage + gq;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              v0r[nt][h] = t0 >= rlo[nt][h] && t0 < rhi[nt][h];
              v1r[nt][h] = t0 + 8 >= rlo[nt][h] && t0 + 8 < rhi[nt][h];
            }
        }
        // A lane's own scores decide whether any running maximum can move
        // this page; only then are the row maxima reduced across the 8 lanes
        // of a row.  Otherwise every maximum stays where it is, which is what
        // the reduction would have decided too.
        float sv[NT][2][2], uv[NT][2][2];   // [tile][row half][token gq, gq + 8]
        bool grow = false;
        // With rows of different lengths in one unit (GEN), a row can meet a
        // page with none of its tokens before any page with one; its maximum
        // is still -inf, and 0 stands in so that exp2 gives 0.
        //
        // The 16-row kernel runs the fp32 steps here and below on packed
        // pairs (the two row halves h of a token; two values per
        // instruction, each rounded as on its own, so the results are those
        // of the scalar form).  The 8-row kernel measured faster scalar.
        constexpr bool kPacked = NT == 2;
        const float2 neg1 = make_float2(-1.f, -1.f);
        if constexpr (kPacked) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float2 a01 = make_float2(sacc[nt][0][0], sacc[nt][0][1]);   // token gq, rows 2c, 2c+1
            float2 a23 = make_float2(sacc[nt][0][2], sacc[nt][0][3]);   // token gq + 8
#pragma unroll
            for (int ch = 1; ch < NCH; ++ch) {
              a01 = __fadd2_rn(a01, make_float2(sacc[nt][ch][0], sacc[nt][ch][1]));
              a23 = __fadd2_rn(a23, make_float2(sacc[nt][ch][2], sacc[nt][ch][3]));
            }
            const float2 s01 = __fmul2_rn(a01, make_float2(fk0, fk0));
            const float2 s23 = __fmul2_rn(a23, make_float2(fk1, fk1));
            sv[nt][0][0] = (GEN ? v0r[nt][0] : v0) ? s01.x : -INFINITY;
            sv[nt][1][0] = (GEN ? v0r[nt][1] : v0) ? s01.y : -INFINITY;
            sv[nt][0][1] = (GEN ? v1r[nt][0] : v1) ? s23.x : -INFINITY;
            sv[nt][1][1] = (GEN ? v1r[nt][1] : v1) ? s23.y : -INFINITY;
            const float2 m2 = make_float2(GEN && m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0],
                                          GEN && m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1]);
            // (s - m_ref) + e_V, s - m_ref as fma(m_ref, -1, s)
            const float2 u0 = __fadd2_rn(__ffma2_rn(m2, neg1, make_float2(sv[nt][0][0], sv[nt][1][0])),
                                         make_float2(evf0, evf0));
            const float2 u1 = __fadd2_rn(__ffma2_rn(m2, neg1, make_float2(sv[nt][0][1], sv[nt][1][1])),
                                         make_float2(evf1, evf1));
            uv[nt][0][0] = u0.x;
            uv[nt][1][0] = u0.y;
            uv[nt][0][1] = u1.x;
            uv[nt][1][1] = u1.y;
            const float2 lazy = make_float2(kLazyMaxLog2, kLazyMaxLog2);
            const float2 mt = __fadd2_rn(make_float2(m_run[nt][0], m_run[nt][1]), lazy);
            const float2 dt = __fadd2_rn(make_float2(d_run[nt][0], d_run[nt][1]), lazy);
            grow |= fmaxf(sv[nt][0][0], sv[nt][0][1]) > mt.x;
            grow |= fmaxf(sv[nt][1][0], sv[nt][1][1]) > mt.y;
            grow |= fmaxf(uv[nt][0][0], uv[nt][0][1]) > dt.x;
            grow |= fmaxf(uv[nt][1][0], uv[nt][1][1]) > dt.y;
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float sres[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float acc = sacc[nt][0][k];
#pragma unroll
              for (int ch = 1; ch < NCH; ++ch) acc += sacc[nt][ch][k];
              sres[k] = acc;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              sv[nt][h][0] = (GEN ? v0r[nt][h] : v0) ? sres[h] * fk0 : -INFINITY;
              sv[nt][h][1] = (GEN ? v1r[nt][h] : v1) ? sres[2 + h] * fk1 : -INFINITY;
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float s0 = sv[nt][h][0], s1 = sv[nt][h][1];
              const float m_ref = GEN && m_run[nt][h] == -INFINITY ? 0.f : m_run[nt][h];
              uv[nt][h][0] = (s0 - m_ref) + evf0;
              uv[nt][h][1] = (s1 - m_ref) + evf1;
              grow |= fmaxf(s0, s1) > m_run[nt][h] + kLazyMaxLog2;
              grow |= fmaxf(uv[nt][h][0], uv[nt][h][1]) > d_run[nt][h] + kLazyMaxLog2;
            }
        }
        bool rescale = false;
        float alpha[NT][2];   // O's factor where the V reference moved
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float tmax = fmaxf(sv[nt][h][0], sv[nt][h][1]);
#pragma unroll
              for (int msk = 4; msk < 32; msk <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, msk));
              const float m_old = m_run[nt][h], d_old = d_run[nt][h];
              const float m_new = tmax > m_old + kLazyMaxLog2 ? tmax : m_old;
              if (!GEN || m_new != m_old) l_run[nt][h] *= fast_exp2(m_old - m_new);
              const float m_ref = GEN && m_new == -INFINITY ? 0.f : m_new;
              uv[nt][h][0] = (sv[nt][h][0] - m_ref) + evf0;
              uv[nt][h][1] = (sv[nt][h][1] - m_ref) + evf1;
              float umax = fmaxf(uv[nt][h][0], uv[nt][h][1]);
#pragma unroll
              for (int msk = 4; msk < 32; msk <<= 1) umax = fmaxf(umax, __shfl_xor_sync(0xffffffffu, umax, msk));
              // the old V reference, relative to the new maximum
              const float d_cur = m_old == -INFINITY ? -INFINITY : d_old + (m_old - m_new);
              const float d_new = umax > d_cur + kLazyMaxLog2 ? umax : d_cur;
              alpha[nt][h] = d_new == d_cur ? 1.f : fast_exp2(d_cur - d_new);
              rescale |= d_new != d_cur;
              m_run[nt][h] = m_new;
              d_run[nt][h] = d_new;
            }
        }
        uint32_t pw[NT][2];
        if constexpr (kPacked) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float2 m2 = make_float2(GEN && m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0],
                                          GEN && m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1]);
            const float2 d2 = make_float2(GEN && d_run[nt][0] == -INFINITY ? 0.f : d_run[nt][0],
                                          GEN && d_run[nt][1] == -INFINITY ? 0.f : d_run[nt][1]);
            const float2 e0 = __ffma2_rn(m2, neg1, make_float2(sv[nt][0][0], sv[nt][1][0]));
            const float2 e1 = __ffma2_rn(m2, neg1, make_float2(sv[nt][0][1], sv[nt][1][1]));
            const float2 x0 = make_float2(fast_exp2(e0.x), fast_exp2(e0.y));
            const float2 x1 = make_float2(fast_exp2(e1.x), fast_exp2(e1.y));
            const float2 l2 = __fadd2_rn(make_float2(l_run[nt][0], l_run[nt][1]), __fadd2_rn(x0, x1));
            l_run[nt][0] = l2.x;
            l_run[nt][1] = l2.y;
            const float2 f0 = __ffma2_rn(d2, neg1, make_float2(uv[nt][0][0], uv[nt][1][0]));
            const float2 f1 = __ffma2_rn(d2, neg1, make_float2(uv[nt][0][1], uv[nt][1][1]));
            pw[nt][0] = movmatrix_trans(pack_f16x2(fast_exp2(f0.x), fast_exp2(f0.y)));
            pw[nt][1] = movmatrix_trans(pack_f16x2(fast_exp2(f1.x), fast_exp2(f1.y)));
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float w4[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float m_ref = GEN && m_run[nt][h] == -INFINITY ? 0.f : m_run[nt][h];
              const float d_ref = GEN && d_run[nt][h] == -INFINITY ? 0.f : d_run[nt][h];
              l_run[nt][h] += fast_exp2(sv[nt][h][0] - m_ref) + fast_exp2(sv[nt][h][1] - m_ref);
              w4[h] = fast_exp2(uv[nt][h][0] - d_ref);
              w4[2 + h] = fast_exp2(uv[nt][h][1] - d_ref);
            }
            pw[nt][0] = movmatrix_trans(pack_f16x2(w4[0], w4[1]));
            pw[nt][1] = movmatrix_trans(pack_f16x2(w4[2], w4[3]));
          }
        }
        if (__any_sync(0xffffffffu, rescale)) {
          if constexpr (Lay::kTmemO) {
            tmem_wait_st();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float oc[32];
              tmem_ld32(o_taddr + 32 * q, oc);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const float a0 = alpha[nt][0], a1 = alpha[nt][1];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  oc[16 * nt + 4 * e] *= a0;
                  oc[16 * nt + 4 * e + 1] *= a1;
                  oc[16 * nt + 4 * e + 2] *= a0;
                  oc[16 * nt + 4 * e + 3] *= a1;
                }
              }
              tmem_st32(o_taddr + 32 * q, oc);
            }
          } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float a0 = alpha[nt][0], a1 = alpha[nt][1];
#pragma unroll
              for (int mt = 0; mt < 16; ++mt) {
                o[nt][mt][0] *= a0;
                o[nt][mt][1] *= a1;
                o[nt][mt][2] *= a0;
                o[nt][mt][3] *= a1;
              }
            }
          }
        }
        // -- PV on the tensor cores
        const uint32_t voff = kVCodeOff + 16 * gq;
        const uint4 va = lds128(sb + ta * kSlotBytes + voff);
        const uint4 vb = lds128(sb + tb * kSlotBytes + voff);
        const uint4 vc = lds128(sb + tcc * kSlotBytes + voff);
        const uint4 vd = lds128(sb + td * kSlotBytes + voff);
        const uint32_t vaw[4] = {va.x, va.y, va.z, va.w}, vbw[4] = {vb.x, vb.y, vb.z, vb.w};
        const uint32_t vcw[4] = {vc.x, vc.y, vc.z, vc.w}, vdw[4] = {vd.x, vd.y, vd.z, vd.w};
        // O^T half h = 2q + nt (columns 16h .. 16h+15) is loaded while the
        // MMAs of half h-1 run; the two halves alternate between ob[0], ob[1].
        float ob[2][16];
        if constexpr (Lay::kTmemO) {
          tmem_wait_st();   // the last page's O^T columns are back
          tmem_ld16_issue(o_taddr, ob[0]);
          tmem_ld16_wait(ob[0]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // pair the same head dim of two tokens in one byte: (token t+1 << 4) | token t
          const uint32_t lo01 = (vaw[q] & 0x0F0F0F0Fu) | ((vbw[q] << 4) & 0xF0F0F0F0u);
          const uint32_t hi01 = ((vaw[q] >> 4) & 0x0F0F0F0Fu) | (vbw[q] & 0xF0F0F0F0u);
          const uint32_t lo89 = (vcw[q] & 0x0F0F0F0Fu) | ((vdw[q] << 4) & 0xF0F0F0F0u);
          const uint32_t hi89 = ((vcw[q] >> 4) & 0x0F0F0F0Fu) | (vdw[q] & 0xF0F0F0F0u);
          uint32_t A0[4], A1[4], A2[4], A3[4];
          f16x2x4_from_e2m1_word(lo01, A0);
          f16x2x4_from_e2m1_word(hi01, A1);
          f16x2x4_from_e2m1_word(lo89, A2);
          f16x2x4_from_e2m1_word(hi89, A3);
          uint32_t a[4][4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            a[e][0] = hmul2(A0[e], rv01);
            a[e][1] = hmul2(A1[e], rv01);
            a[e][2] = hmul2(A2[e], rv89);
            a[e][3] = hmul2(A3[e], rv89);
          }
          if constexpr (Lay::kTmemO) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const int h = 2 * q + nt, cur = h & 1;
              if (h < 7) tmem_ld16_issue(o_taddr + 16 * (h + 1), ob[cur ^ 1]);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                mma_f16_16816(*reinterpret_cast<float(*)[4]>(ob[cur] + 4 * e), a[e][0], a[e][1], a[e][2],
                              a[e][3], pw[nt][0], pw[nt][1]);
              tmem_st16(o_taddr + 16 * h, ob[cur]);
              if (h < 7) tmem_ld16_wait(ob[cur ^ 1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_f16_16816(o[nt][4 * q + e], a[e][0], a[e][1], a[e][2], a[e][3], pw[nt][0], pw[nt][1]);
          }
        }
      }
      __syncwarp();
      if (j + NSTAGE < n_my) issue(j + NSTAGE, stg);   // same stage, next phase
      if (++stg == NSTAGE) {
        stg = 0;
        phase ^= 1u;
      }
    }
    if (timed_out) {
      if (lane == 0) atomicOr(err, kErrTimeout);
      // wait (bounded) for this warp's copies still in flight, then stop the CTA
      for (int jj = j; jj < n_my && jj < j + NSTAGE; ++jj) {
        (void)mbar_wait(bar_base + 8 * stg, phase);
        if (++stg == NSTAGE) {
          stg = 0;
          phase ^= 1u;
        }
      }
      s_misc[1] = 1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          m_run[nt][h] = -INFINITY;
          d_run[nt][h] = -INFINITY;
          l_run[nt][h] = 0.f;
        }
    }
    tiles_done += (uint32_t)n_my;
    // full row sums over the 8 lanes that share c
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1)
          l_run[nt][h] += __shfl_xor_sync(0xffffffffu, l_run[nt][h], msk);

    // ---- merge the warps' states: partial (o, lse) of this split ---------------
    __syncthreads();  // every warp is done with its stage buffers
    float* osm = reinterpret_cast<float*>(smem);
    float* stats = reinterpret_cast<float*>(smem + Lay::kStatsOff);
    float* rowinfo = reinterpret_cast<float*>(smem + Lay::kRowInfoOff);
    float* my_o = osm + warp * Lay::kRows * Lay::kORowStride;
    if (gq == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float* st = stats + (warp * Lay::kRows + nt * 8 + 2 * c + h) * 4;
          st[0] = m_run[nt][h];
          st[1] = d_run[nt][h];
          st[2] = l_run[nt][h];
        }
    }
    // The next unit is taken now; its word is read during the merge below.
    // A CTA that gave up (its abort flag is set before the merge barriers)
    // takes no more, so that no unit is taken and then left undone.
    int next_u = n_units;
    if (threadIdx.x == 0 && !s_misc[1]) next_u = atomicAdd(&ws.hdr[1], 1);
    __syncthreads();
    const int out_rows = QG * pack;   // rows 0 .. out_rows-1 may be written
    // output row (sequence or chunk position, query head) of unit row r
    auto out_row = [&](int r) {
      return GEN ? (int64_t)row_of(r) * Hq + head_of(r) : (int64_t)(b * Hq + g * QG + r);
    };
    if (threadIdx.x < out_rows && (!GEN || row_exists(threadIdx.x))) {
      const int r = threadIdx.x;
      const int64_t orow = out_row(r);
      float M = -INFINITY;
      for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, stats[(w * Lay::kRows + r) * 4]);
      float Ls = 0.f;
      bool bad = false;   // a warp met a token beyond the f16 span: the exact pass redoes the unit
      for (int w = 0; w < NWARPS; ++w) {
        const float* st = stats + (w * Lay::kRows + r) * 4;
        if (st[2] > 0.f) Ls += st[2] * fast_exp2(st[0] - M);
        bad |= isnan(st[2]);
      }
      if (bad) s_misc[3] = 1;
      float* ri = rowinfo + r * (NWARPS + 2);
      for (int w = 0; w < NWARPS; ++w) {
        const float* st = stats + (w * Lay::kRows + r) * 4;
        ri[w] = (Ls > 0.f && st[2] > 0.f) ? fast_exp2((st[0] - M) + st[1]) / Ls : 0.f;
      }
      ri[NWARPS] = Ls > 0.f ? M + fast_log2(Ls) : -INFINITY;
      ws.part_lse[orow * S + split] = ri[NWARPS];
    }
    // the next unit's work-list word, in flight while the parts are merged
    int next_word = 0;
    if (threadIdx.x == 0 && next_u < n_units) next_word = (int)ws.units[next_u];
    // Lane (gq, c) holds head dims 32gq .. 32gq+31 of rows nt*8 + 2c (+1);
    // the head dims are merged in kMergeParts parts through one buffer.
#pragma unroll
    for (int part = 0; part < Lay::kMergeParts; ++part) {
      const bool mine = (32 * gq) / Lay::kPartDims == part;
      const int dbase = 32 * gq - part * Lay::kPartDims;
      if constexpr (Lay::kTmemO) {
        tmem_wait_st();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float oc[32];
          tmem_ld32(o_taddr + 32 * q, oc);
          if (mine) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const int r0 = nt * 8 + 2 * c;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float* v = oc + 16 * nt + 4 * e;
                const int d = dbase + 2 * (4 * q + e);
                *reinterpret_cast<float2*>(my_o + r0 * Lay::kORowStride + d) = make_float2(v[0], v[2]);
                *reinterpret_cast<float2*>(my_o + (r0 + 1) * Lay::kORowStride + d) = make_float2(v[1], v[3]);
              }
            }
          }
        }
      } else if (mine) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int r0 = nt * 8 + 2 * c;
#pragma unroll
          for (int mt = 0; mt < 16; ++mt) {
            const int d = dbase + 2 * mt;
            *reinterpret_cast<float2*>(my_o + r0 * Lay::kORowStride + d) = make_float2(o[nt][mt][0], o[nt][mt][2]);
            *reinterpret_cast<float2*>(my_o + (r0 + 1) * Lay::kORowStride + d) = make_float2(o[nt][mt][1], o[nt][mt][3]);
          }
        }
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < out_rows * (Lay::kPartDims / 4); idx += NWARPS * 32) {
        const int r = idx / (Lay::kPartDims / 4), d4 = (idx % (Lay::kPartDims / 4)) * 4;
        if (GEN && !row_exists(r)) continue;
        const int64_t orow = out_row(r);
        const float* ri = rowinfo + r * (NWARPS + 2);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) {
          const float f = ri[w];
          const float4 v = *reinterpret_cast<const float4*>(osm + (w * Lay::kRows + r) * Lay::kORowStride + d4);
          acc.x += v.x * f;
          acc.y += v.y * f;
          acc.z += v.z * f;
          acc.w += v.w * f;
        }
        *reinterpret_cast<float4*>(ws.part_o + (orow * S + split) * kHeadDim + part * Lay::kPartDims + d4) = acc;
      }
      __syncthreads();  // the merge buffer (the stage buffers) and Q' are free again
    }
    if (threadIdx.x == 0) {
      if (s_misc[3]) {
        ws.redo[atomicAdd(&ws.hdr[2], 1)] = (uint32_t)u;
        s_misc[3] = 0;
      }
      s_misc[5] = next_u;
      s_misc[6] = next_word;
    }
  }
  if constexpr (Lay::kTmemO) {
    tmem_wait_st();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc((uint32_t)s_misc[2], kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// The exact pass: the units that stage 1 listed for a redo (a token whose K
// blocks span 2^28 or more) are recomputed in plain fp32, one warp per unit
// over all of its pages, and their split partials are overwritten before
// stage 2 merges them.  With an empty list every CTA returns at once.
// ---------------------------------------------------------------------------
constexpr int kExactWarps = 4;

template <bool GEN>
__global__ void __launch_bounds__(kExactWarps * 32)
decode_exact_units(const uint16_t* __restrict__ query, int64_t q_ss, int64_t q_sh, const uint8_t* __restrict__ kv,
                   const int32_t* __restrict__ block_table, const SeqRows rows, float scale_log2e, int Hq, int Hk,
                   int QG, int num_blocks, int S, Workspace ws) {
  __shared__ __align__(16) uint16_t q_all[kExactWarps][16][kHeadDim];   // q' of each warp's unit rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  pdl_launch_dependents();
  pdl_wait();   // stage 1's partials and redo list are complete
  const int n = ws.hdr[2];
  for (int i = blockIdx.x * kExactWarps + warp; i < n; i += gridDim.x * kExactWarps) {
    const uint32_t unit = ws.units[ws.redo[i]];
    const int b = (int)(unit & 0xffffu), split = (int)((unit >> 16) & 0xffu), g = (int)(unit >> 24);
    // the unit's rows and pages, derived as in stage 1
    const int L = GEN ? unit_len(rows, b) : row_len(rows, b);
    const int P = (L + kPage - 1) / kPage;
    const int lo = GEN ? unit_lo(rows, b) : 0;
    const int pack = GEN ? rows.pack : 1;
    const int last_row = GEN ? unit_last_row(rows, b) : b;
    auto row_of = [&](int r) { return GEN ? min(b * pack + r / QG, last_row) : b; };
    auto row_exists = [&](int r) { return GEN ? r < QG * pack && b * pack + r / QG <= last_row : r < QG; };
    auto head_of = [&](int r) { return g * QG + (GEN ? r % QG : r); };
    const int p_begin = lo / kPage + split * ws.seq_info[b].x;
    const int p_end = min(p_begin + ws.seq_info[b].x, P);
    const int out_rows = QG * pack;   // <= 16
    uint16_t(*qw)[kHeadDim] = q_all[warp];
    for (int r = 0; r < 16; ++r) {
      uint32_t pk[4] = {0u, 0u, 0u, 0u};
      if (r < out_rows && row_exists(r))
        query_prime8(query + (int64_t)row_of(r) * q_ss + (int64_t)head_of(r) * q_sh, lane, pk);
      *reinterpret_cast<uint4*>(&qw[r][8 * lane]) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    __syncwarp();
    const int32_t* bt_row = block_table + (int64_t)b * rows.bt_stride;
    const int lg_tpp = GEN ? rows.lg_tpp : 0;
    for (int nt = 0; nt * 8 < out_rows; ++nt) {
      int rlo[2] = {0, 0}, rhi[2] = {L, L};
      if constexpr (GEN) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          rhi[h] = row_len(rows, row_of(nt * 8 + 2 * c + h));
          rlo[h] = row_lo(rows, rhi[h]);
        }
      }
      float m[2], d[2], l[2], acc[16][4];
      exact_rows<GEN>(kv, bt_row, num_blocks, Hk, g, lg_tpp, p_begin, p_end - p_begin, 1, L, rlo, rhi,
                      reinterpret_cast<const uint8_t*>(&qw[nt * 8 + 2 * c][0]), kHeadDim * 2, scale_log2e, gq, m,
                      d, l, acc);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], msk);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = nt * 8 + 2 * c + h;
        if (r >= out_rows || (GEN && !row_exists(r))) continue;
        const int64_t orow = GEN ? (int64_t)row_of(r) * Hq + head_of(r) : (int64_t)(b * Hq + g * QG + r);
        const float fac = l[h] > 0.f ? exp2f(d[h]) / l[h] : 0.f;
        if (gq == 0) ws.part_lse[orow * S + split] = l[h] > 0.f ? m[h] + log2f(l[h]) : -INFINITY;
        float* dst = ws.part_o + (orow * S + split) * kHeadDim + 32 * gq;
#pragma unroll
        for (int mt = 0; mt < 16; ++mt)
          *reinterpret_cast<float2*>(dst + 2 * mt) = make_float2(acc[mt][h] * fac, acc[mt][2 + h] * fac);
      }
    }
    __syncwarp();   // q_all[warp] is rewritten by the warp's next unit
  }
}

// ---------------------------------------------------------------------------
// Stage 2: merge the active splits of each (sequence, query head).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
decode_stage2(Workspace ws, int B, int Hq, int S, int pack, const float* __restrict__ sinks,
              uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  pdl_wait();   // stage 1's partials are complete
  if (row >= B * Hq) return;
  const int b = row / Hq;
  const int n = ws.seq_info[b / pack].y;   // row b's unit row holds its split count
  const float* lse = ws.part_lse + (int64_t)row * S;
  const float* po = ws.part_o + (int64_t)row * S * kHeadDim + lane * 8;
  // The first 32 splits' log-sum-exps are loaded before the split count
  // arrives (slots past it hold stale words and are never used), and the
  // first kSpec splits' partials all at once as soon as it has, so a row's
  // reads take two round trips instead of a chain.
  constexpr int kSpec = 8;
  const float lse_lane = lane < S ? lse[lane] : -INFINITY;
  float4 vs[kSpec][2];
#pragma unroll
  for (int i = 0; i < kSpec; ++i) {
    if (i < n) {
      vs[i][0] = *reinterpret_cast<const float4*>(po + (int64_t)i * kHeadDim);
      vs[i][1] = *reinterpret_cast<const float4*>(po + (int64_t)i * kHeadDim + 4);
    }
  }
  float mx = lane < n ? lse_lane : -INFINITY;
  for (int s = lane + 32; s < n; s += 32) mx = fmaxf(mx, lse[s]);
#pragma unroll
  for (int msk = 16; msk > 0; msk >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
  // a sink logit joins the denominator only (log2 units like the partials)
  const float zs = sinks ? sinks[row % Hq] * kLog2e : -INFINITY;
  mx = fmaxf(mx, zs);
  // the denominator first, so that each split enters the sum already
  // weighted by its share (<= 1): the running sum never exceeds the largest
  // split output in magnitude, even next to fp32's top
  float den = 0.f;
  if (mx > -INFINITY) {
    if (lane < n) den += fast_exp2(lse_lane - mx);
    for (int s = lane + 32; s < n; s += 32) den += fast_exp2(lse[s] - mx);
  }
#pragma unroll
  for (int msk = 16; msk > 0; msk >>= 1) den += __shfl_xor_sync(0xffffffffu, den, msk);
  if (zs > -INFINITY) den += fast_exp2(zs - mx);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (n > 0 && mx > -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      const float wl = (s0 + lane < n) ? fast_exp2((s0 == 0 ? lse_lane : lse[s0 + lane]) - mx) * inv : 0.f;
      const int cnt = min(32, n - s0);
      auto add = [&](int k, const float4& v0, const float4& v1) {
        const float w = __shfl_sync(0xffffffffu, wl, k);
        acc[0] += w * v0.x; acc[1] += w * v0.y; acc[2] += w * v0.z; acc[3] += w * v0.w;
        acc[4] += w * v1.x; acc[5] += w * v1.y; acc[6] += w * v1.z; acc[7] += w * v1.w;
      };
      int k = 0;
      if (s0 == 0) {
#pragma unroll
        for (int i = 0; i < kSpec; ++i)
          if (i < cnt) add(i, vs[i][0], vs[i][1]);
        k = kSpec;
      }
      // later splits: four partials are loaded before any is used, so
      // their latencies overlap; the sums keep the split order
      for (; k + 4 <= cnt; k += 4) {
        float4 v[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float* pp = po + (int64_t)(s0 + k + i) * kHeadDim;
          v[i][0] = *reinterpret_cast<const float4*>(pp);
          v[i][1] = *reinterpret_cast<const float4*>(pp + 4);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) add(k + i, v[i][0], v[i][1]);
      }
      for (; k < cnt; ++k) {
        const float* pp = po + (int64_t)(s0 + k) * kHeadDim;
        add(k, *reinterpret_cast<const float4*>(pp), *reinterpret_cast<const float4*>(pp + 4));
      }
    }
  }
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(acc[2 * i + 1]), "f"(acc[2 * i]));
    pk[i] = r;
  }
  *reinterpret_cast<uint4*>(out + (int64_t)row * kHeadDim + lane * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
// Record a caller's timing event.  Under stream capture a plain record only
// becomes a dependency edge, so it is captured as an external event node.
static cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
             : cudaEventRecord(ev, stream);
}

// Launch `kern` so that it may start while the previous kernel on the
// stream finishes (programmatic stream serialization); the kernel waits in
// pdl_wait before it reads that kernel's results.
template <typename... Params, typename... Args>
static cudaError_t launch_overlapped(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Per device, context and instantiation: set the shared-memory opt-in once
// and size the persistent grid from the occupancy the kernel actually gets.
// The cache is shared by all host threads, under a lock.
cudaError_t current_context_id(unsigned long long* id);
static std::mutex g_grid_mutex;

template <int NT, int GEN>
static cudaError_t stage1_grid(int* grid) {
  constexpr int NWARPS = 4, NSTAGE = kStage1Stages;
  using Lay = Stage1Layout<NT, NWARPS, NSTAGE>;
  static int grid_of_device[64] = {0};
  static unsigned long long ctx_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned long long ctx = 0;
  if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_grid_mutex);
  if (dev >= 0 && dev < 64 && grid_of_device[dev] > 0 && ctx_of_device[dev] == ctx) {
    *grid = grid_of_device[dev];
    return cudaSuccess;
  }
  auto kern = decode_stage1<NT, NWARPS, NSTAGE, GEN>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if constexpr (Lay::kTmemO) {
    // The occupancy query does not model a kernel that allocates tensor
    // memory, so count the limits directly: registers per scheduler (one
    // warp of each CTA per scheduler), shared memory, and the 512 TMEM
    // columns of an SM.
    cudaFuncAttributes fa;
    int smem_sm = 0, reserved = 0;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
      return e;
    const int regs = (fa.numRegs + 7) & ~7;
    const int by_regs = regs > 0 ? 16384 / (regs * 32) : 1;
    const int by_smem = smem_sm / (Lay::kBytes + reserved);
    per_sm = by_regs < by_smem ? by_regs : by_smem;
    if (per_sm > (int)(512 / kTmemCols)) per_sm = (int)(512 / kTmemCols);
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NWARPS * 32, Lay::kBytes);
    if (e != cudaSuccess) return e;
  }
  *grid = sms * (per_sm > 0 ? per_sm : 1);
  if (dev >= 0 && dev < 64) {
    grid_of_device[dev] = *grid;
    ctx_of_device[dev] = ctx;
  }
  return cudaSuccess;
}

// The cache as a 3-D tensor of 32-bit words: x = word within a slot (68),
// y = kv head (Hk, stride 272 B), z = slot (num_blocks * block_size, stride
// Hk * 272 B).  One box of 68 x 1 x 16 words is one (16-token tile, kv head).
cudaError_t make_kv_tensor_map(CUtensorMap* map, const uint8_t* kv, int Hk, int64_t num_slots) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  static cudaError_t lookup = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    lookup = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (lookup == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) lookup = cudaErrorNotSupported;
    if (lookup == cudaSuccess) encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (lookup != cudaSuccess) return lookup;
  const cuuint64_t dims[3] = {kSlotBytes / 4, (cuuint64_t)Hk, (cuuint64_t)num_slots};
  const cuuint64_t strides[2] = {kSlotBytes, (cuuint64_t)Hk * kSlotBytes};
  const cuuint32_t box[3] = {kSlotBytes / 4, 1, kPage};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(kv), dims,
                      strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      static_cast<CUtensorMapL2promotion>(UQ_KV_L2_PROMOTION), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Plan, then stage 1 (bracketed by the caller's timing events, if any).
template <int NT, int GEN>
static cudaError_t launch_plan_and_stage1(const uint16_t* query, int64_t q_ss, int64_t q_sh,
                                          const uint8_t* kv, const int32_t* bt, const SeqRows& sl,
                                          float scale, int B, int Hq, int Hk, int num_blocks,
                                          int max_blocks, int S, const Workspace& ws, unsigned* err,
                                          cudaStream_t stream, cudaEvent_t ev_before,
                                          cudaEvent_t ev_after) {
  constexpr int NWARPS = 4, NSTAGE = kStage1Stages;
  using Lay = Stage1Layout<NT, NWARPS, NSTAGE>;
  int grid = 0;
  cudaError_t e = stage1_grid<NT, GEN>(&grid);
  if (e != cudaSuccess) return e;
  CUtensorMap kv_map;
  const int64_t num_slots = (int64_t)num_blocks << (4 + sl.lg_tpp);
  if ((e = make_kv_tensor_map(&kv_map, kv, Hk, num_slots)) != cudaSuccess) return e;
  e = launch_overlapped(decode_plan, dim3(1), dim3(kPlanThreads), 0, stream, sl, (B + sl.pack - 1) / sl.pack, Hk,
                        S, grid, NT == 2 ? kUnitCostTiles16 : kUnitCostTiles8, ws);
  if (e != cudaSuccess) return e;
  if (ev_before && (e = record_timing_event(ev_before, stream)) != cudaSuccess) return e;
  e = launch_overlapped(decode_stage1<NT, NWARPS, NSTAGE, GEN>, dim3(grid), dim3(NWARPS * 32), Lay::kBytes,
                        stream, query, q_ss, q_sh, kv_map, kv, bt, sl, scale * kLog2e, Hq, Hk, Hq / Hk,
                        num_blocks, S, ws, err);
  if (e != cudaSuccess) return e;
  if (ev_after && (e = record_timing_event(ev_after, stream)) != cudaSuccess) return e;
  return launch_overlapped(decode_exact_units<(GEN != 0)>, dim3((grid + 3) / 4), dim3(kExactWarps * 32), 0, stream, query,
                           q_ss, q_sh, kv, bt, sl, scale * kLog2e, Hq, Hk, Hq / Hk, num_blocks, S, ws);
}

size_t decode_workspace_bytes(int B, int Hq, int S) { return workspace_bytes(B, Hq, S); }

cudaError_t launch_decode(const uint16_t* query, int64_t q_ss, int64_t q_sh, const uint8_t* kv,
                          const int32_t* bt, const SeqRows& sl, float scale, const float* sinks,
                          int B, int Hq, int Hk, int num_blocks, int max_blocks, int S,
                          void* workspace, uint16_t* out, unsigned* err, cudaStream_t stream,
                          cudaEvent_t ev_before_stage1, cudaEvent_t ev_after_stage1) {
  const Workspace ws = workspace_layout(workspace, B, Hq, S);
  // 2: a window or pages of more than 16 tokens; 1: multi-query unit rows only
  const int gen = (sl.window > 0 || sl.lg_tpp > 0) ? 2 : (sl.pack > 1 ? 1 : 0);
  const bool sixteen = (Hq / Hk) * sl.pack > 8;
  auto run = [&](auto nt, auto g) {
    return launch_plan_and_stage1<decltype(nt)::value, decltype(g)::value>(
        query, q_ss, q_sh, kv, bt, sl, scale, B, Hq, Hk, num_blocks, max_blocks, S, ws, err, stream,
        ev_before_stage1, ev_after_stage1);
  };
  using One = std::integral_constant<int, 1>;
  using Two = std::integral_constant<int, 2>;
  using Plain = std::integral_constant<int, 0>;
  using MqRows = std::integral_constant<int, 1>;
  using Gen = std::integral_constant<int, 2>;
  // 8-row units never hold two chunk positions (6- and 8-row groups pack
  // into 16-row units), so they take the general kernel for any GEN case
  cudaError_t e = sixteen ? (gen == 2 ? run(Two{}, Gen{}) : gen == 1 ? run(Two{}, MqRows{}) : run(Two{}, Plain{}))
                          : (gen != 0 ? run(One{}, Gen{}) : run(One{}, Plain{}));
  if (e != cudaSuccess) return e;
  const int rows = B * Hq;
  return launch_overlapped(decode_stage2, dim3((rows + 3) / 4), dim3(128), 0, stream, ws, B, Hq, S, sl.pack,
                           sinks, out);
}

}  // namespace uq
