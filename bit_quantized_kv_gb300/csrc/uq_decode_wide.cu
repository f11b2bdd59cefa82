// uq_decode_wide.cu -- stage 1 of the split-KV decode for work units of 16
// to 64 query rows (16 query heads per kv head, or the query heads of several
// positions of a continuation chunk), on the 5th-generation tensor cores.
// (vllm.v1.attention.ops.flydsl_ultraquant_decode: QK as a scaled FP4 x E4M3
// product with the UE8M0 K scales applied by the tensor core, PV with the V
// codes converted natively; its partition partials and their reduce.)
//
// A work unit is (unit row, split, kv head) from the same device-side plan
// as the other stage-1 kernel; it is walked in groups of 128 tokens (8 tiles
// of 16 tokens).  One persistent CTA per SM, ten warps in four roles:
//
//   warp 0      producer: takes units from the plan's counter, publishes
//               them in a 4-deep ring, and copies each tile (16 slots of one
//               kv head, 4352 bytes) into a ring of stage buffers with one
//               TMA tensor copy completing on that buffer's mbarrier.
//   warp 1      one thread issues every tensor-core instruction:
//               QK  S[128 tokens x NR rows] = K (E2M1 codes, UE8M0 block
//                   scales in tensor memory) x q' (E4M3), eight block-scaled
//                   MMAs per group (kind::mxf8f6f4, one 32-element block of
//                   the head dimension each), into tensor memory;
//               PV  O^T[256 dims x NR rows] += V'^T[dims x 128 tokens] x
//                   P^T[tokens x rows], V'^T read from tensor memory, P^T
//                   from shared memory (kind::f16, fp32 accumulation), 16
//                   MMAs per group (two halves of 128 dims, K = 16 tokens).
//   warps 2-5   convert, one per tensor-memory lane quarter q: the K codes of
//               tiles 2q, 2q+1 into the padded E2M1 operand layout (16-element
//               chunks of 8 code bytes and 8 unused bytes), their K scales
//               into tensor memory, and for every tile of the group the V
//               codes of head dims 64q .. 64q+63 as f16 V' = c * 2^(13 + e -
//               E_t) (E_t the token's largest V block exponent) straight into
//               the PV A operand in tensor memory, from registers laid out as
//               the mma.m16n8k16 A fragment (tcgen05.st 16x128b).
//   warps 6-9   softmax, one per lane quarter: lane = token of the group.
//               Scores come out of tensor memory; a lazy running maximum m
//               and a V reference d relative to it (both per row, in shared
//               memory) move only when a group exceeds them by more than 2^8,
//               decided by one OR-vote of the four warps; P^T (f16) goes to
//               shared memory; the rare rescale of O^T runs in tensor memory.
//               At the end of a unit the four warps merge the row sums and
//               write the split partial (normalised O, log2-sum-exp).
//
// Per token t and row r (log2 units): s = scale*log2(e) * q'.k_t, exactly
// scaled by the tensor core; p = 2^(s - m) sums into l; the PV weight is
// w = 2^((s - m) + e_t - d), e_t = E_t - 127 - 13, so that w * V'_t =
// 2^(s - m - d) V_t and the partial is O * 2^d / l with lse = m + log2 l.
//
// Every wait on an mbarrier is bounded; when one runs out the CTA records
// UQ_DEVERR_TIMEOUT, raises an abort flag that every role polls, drains the
// copies and tensor-core work it has in flight, and ends.  The softmax warps
// combine the outcome of their waits in an OR-vote before each named barrier
// they share, so they always leave together.
#include <mutex>

#include "uq_decode_common.cuh"

namespace uq {
namespace wide {

constexpr int kWarps = 10;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kSoftWarp0 = 6;   // warps 2-5 convert
constexpr int kGroupTiles = 8;
constexpr int kGroupTokens = kGroupTiles * kPage;     // 128: M of the QK MMA
constexpr int kKaChunk = kGroupTokens / 8 * 128;      // K operand: stride between 16-element chunks
constexpr int kKaBytes = kGroupTokens * kHeadDim;     // 32 KB: 256 padded code bytes per token
constexpr int kPbNGroup = kGroupTokens / 8 * 128;     // P^T operand: stride between 8-row groups
constexpr uint32_t kSoftBar = 1;                      // named barrier of the four softmax warps
constexpr uint32_t kSoftThreads = 128;
constexpr uint32_t kTmemCols = 512;

// Scores of one chunk of rows (16 or 32 columns) for the thread's token lane.
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[16]) { tmem_ld16(taddr, v); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[32]) { tmem_ld32(taddr, v); }

template <int NR>
struct Layout {
  static_assert(NR == 16 || NR == 32 || NR == 64, "query rows per unit");
  static constexpr int kNS = NR <= 32 ? 2 : 1;            // score buffers in tensor memory
  static constexpr int kStageTiles = NR <= 32 ? 24 : 16;  // TMA ring, tiles
  // shared memory
  static constexpr int kKaOff = (kStageTiles * kTileBytes + 1023) / 1024 * 1024;   // [2] K operand
  static constexpr int kQbOff = kKaOff + 2 * kKaBytes;    // q' operand, E4M3 [NR][256]
  static constexpr int kQbChunk = NR / 8 * 128;           // its stride between 16-dim chunks
  static constexpr int kPbOff = kQbOff + NR * kHeadDim;   // [2] P^T operand, f16
  static constexpr int kPbBytes = kGroupTokens * NR * 2;
  static constexpr int kEvfOff = kPbOff + 2 * kPbBytes;   // [2][128] fp32 V exponent e_t
  static constexpr int kGnvOff = kEvfOff + 2 * kGroupTokens * 4;   // [2][8] valid tokens per tile
  static constexpr int kSnvOff = kGnvOff + 2 * kGroupTiles * 4;    // [stage] valid tokens
  static constexpr int kMetaOff = kSnvOff + kStageTiles * 4;       // [4 warps][128 tokens] f16x2
  static constexpr int kRowOff = kMetaOff + 4 * kGroupTokens * 4;  // rlo[NR], rhi[NR]
  static constexpr int kStatOff = kRowOff + 2 * NR * 4;            // m[NR], d[NR]
  static constexpr int kRedOff = kStatOff + 2 * NR * 4;            // [4][2][NR] scratch
  static constexpr int kFacOff = kRedOff + 4 * 2 * NR * 4;         // [NR] factors
  static constexpr int kUnitOff = kFacOff + NR * 4;                // [4] unit ring
  static constexpr int kMiscOff = kUnitOff + 16;                   // [0] abort, [1] TMEM base, [2] units done
  static constexpr int kBarOff = kMiscOff + 16;
  // mbarriers
  static constexpr int bFull = 0;
  static constexpr int bEmpty = bFull + kStageTiles;
  static constexpr int bConv = bEmpty + kStageTiles;   // [2]
  static constexpr int bKaFree = bConv + 2;            // [2]
  static constexpr int bPvDone = bKaFree + 2;          // [2]
  static constexpr int bSFull = bPvDone + 2;           // [kNS]
  static constexpr int bSFree = bSFull + kNS;          // [kNS]
  static constexpr int bPFull = bSFree + kNS;          // [2]
  static constexpr int bQFull = bPFull + 2;
  static constexpr int bUFull = bQFull + 1;            // [4]
  static constexpr int bUEmpty = bUFull + 4;           // [4]
  static constexpr int kNumBars = bUEmpty + 4;
  static constexpr int kBytes = kBarOff + kNumBars * 8;
  // tensor memory columns
  static constexpr uint32_t kTmVt = 0;                  // [buf][half] 64 columns: V'^T
  static constexpr uint32_t kTmO = 256;                 // [half] NR columns: O^T
  static constexpr uint32_t kTmS = (kTmO + 2 * NR + 31) / 32 * 32;   // [kNS] NR columns: S
  static constexpr uint32_t kTmSfa = kTmS + kNS * NR;   // [buf] 8 columns: K block scales
  static constexpr uint32_t kTmSfb = kTmSfa + 16;       // 8 columns: q' scales (2^0)
  static_assert(kTmSfb + 8 <= kTmemCols, "tensor memory");
  static_assert(kBytes <= 227 * 1024, "shared memory");
};

struct Unit {
  int b, split, g, L, p_begin, n_tiles, n_groups;
};

__device__ __forceinline__ Unit decode_unit(const SeqRows& rows, const Workspace& ws, int u) {
  const uint32_t e = ws.units[u];
  Unit t;
  t.b = (int)(e & 0xffffu);
  t.split = (int)((e >> 16) & 0xffu);
  t.g = (int)(e >> 24);
  t.L = unit_len(rows, t.b);
  const int pps = ws.seq_info[t.b].x;
  const int P = (t.L + kPage - 1) / kPage;
  t.p_begin = unit_lo(rows, t.b) / kPage + t.split * pps;
  t.n_tiles = max(0, min(t.p_begin + pps, P) - t.p_begin);
  t.n_groups = (t.n_tiles + kGroupTiles - 1) / kGroupTiles;
  return t;
}

// Bounded wait for the phase of `bar` with the given parity.  Gives up early
// when another role raised the abort flag; on running out it raises the flag
// and records the timeout.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* err) {
  for (uint32_t it = 0; it < kWaitSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(kWaitSuspendNs) : "memory");
    if (done) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
  return false;
}

// The same, taken by every lane of the warp: true only if all lanes saw the
// phase complete, so that the warp's collective instructions stay converged.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err));
}

// Non-blocking test of a phase, taken by the whole warp (true only if every
// lane saw it complete).
__device__ __forceinline__ bool test_warp(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return __all_sync(0xffffffffu, done != 0);
}

// One short suspended wait for a phase (returns when it completes or after
// about kPollNs); the caller re-tests what it is waiting for.  kPollLimit
// such polls take about as long as one full bounded wait.
constexpr uint32_t kPollNs = 256;
constexpr uint32_t kPollLimit = kWaitSpinLimit * (kWaitSuspendNs > kPollNs ? kWaitSuspendNs / kPollNs : 1u);
__device__ __forceinline__ void poll_bar(uint32_t bar, uint32_t parity) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%0], %1, %2;\n}\n"
      :: "r"(bar), "r"(parity), "r"(kPollNs) : "memory");
}

// Head dim held by tensor-memory lane `l` (0..31) of quarter q in half h of
// the PV operands: the convert warps place dims 64q + 8g + 4h + 2mt + r at
// lane 16mt + 8r + g (g = 0..7, mt, r = 0..1).
__device__ __forceinline__ int lane_dim(int q, int h, int l) {
  return 64 * q + 8 * (l & 7) + 4 * h + 2 * (l >> 4) + ((l >> 3) & 1);
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1)
decode_stage1_wide(const uint16_t* __restrict__ query, int64_t q_ss, int64_t q_sh,
                   const __grid_constant__ CUtensorMap kv_map, const int32_t* __restrict__ block_table,
                   const SeqRows rows, float scale_log2e, int Hq, int Hk, int num_blocks, int S,
                   Workspace ws, unsigned* __restrict__ err) {
  using Lay = Layout<NR>;
  constexpr int kChunk = NR < 32 ? NR : 32;   // softmax rows per tensor-memory load
  constexpr int KST = Lay::kStageTiles;
  constexpr int NS = Lay::kNS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + Lay::kMiscOff);
  volatile int* s_unit = reinterpret_cast<volatile int*>(smem + Lay::kUnitOff);
  volatile int* abort_flag = misc;
  auto bar = [&](int i) { return sbase + Lay::kBarOff + 8u * (uint32_t)i; };
  auto stage = [&](uint32_t slot) { return sbase + slot * (uint32_t)kTileBytes; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < KST; ++i) {
      mbar_init(bar(Lay::bFull + i), 1);
      mbar_init(bar(Lay::bEmpty + i), 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Lay::bConv + i), 4);
      mbar_init(bar(Lay::bKaFree + i), 1);
      mbar_init(bar(Lay::bPvDone + i), 1);
      mbar_init(bar(Lay::bPFull + i), 4);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(Lay::bSFull + i), 1);
      mbar_init(bar(Lay::bSFree + i), 4);
    }
    mbar_init(bar(Lay::bQFull), 4);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(Lay::bUFull + i), 1);
      mbar_init(bar(Lay::bUEmpty + i), 9);
    }
    misc[0] = 0;
    misc[2] = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(sbase + Lay::kMiscOff + 4, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = (uint32_t)misc[1];

  pdl_launch_dependents();   // stage 2 may be scheduled as CTAs retire
  pdl_wait();                // the plan's work list is complete
  const int n_units = ws.hdr[0];
  const int QG = Hq / Hk;

  int published = 0, pending = -1;   // producer: units handed to the ring; one taken but not handed
  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&kv_map)) : "memory");
    uint32_t tc = 0;
    const int lg = rows.lg_tpp, tmask = (1 << lg) - 1;
    for (;;) {
      int u = 0;
      if (lane == 0) u = atomicAdd(&ws.hdr[1], 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      const int us = published & 3;
      if (!wait_warp(bar(Lay::bUEmpty + us), ((published >> 2) & 1) ^ 1, abort_flag, err)) {
        pending = u < n_units ? u : -1;
        break;
      }
      const bool stop = u >= n_units || *abort_flag;
      if (lane == 0) {
        s_unit[us] = stop ? -1 : u;
        mbar_arrive(bar(Lay::bUFull + us));
      }
      if (stop) {
        pending = u < n_units ? u : -1;
        break;
      }
      ++published;
      const Unit U = decode_unit(rows, ws, u);
      const int32_t* bt_row = block_table + (int64_t)U.b * rows.bt_stride;
      // A group of up to 8 tiles at a time: lane i waits for its tile's stage
      // buffer and issues that tile's copy, so the copies of a group leave
      // together; the page ids of the next group are loaded a group ahead.
      bool aborted = false;
      int pid_next = lane < min(kGroupTiles, U.n_tiles) ? bt_row[(U.p_begin + lane) >> lg] : -1;
      for (int j0 = 0; j0 < U.n_tiles; j0 += kGroupTiles) {
        const int n_here = min(kGroupTiles, U.n_tiles - j0);
        const int pid = pid_next;
        const int jn = j0 + kGroupTiles + lane;
        pid_next = (lane < kGroupTiles && jn < U.n_tiles) ? bt_row[(U.p_begin + jn) >> lg] : -1;
        const uint32_t t_i = tc + (uint32_t)lane, slot = t_i % KST;
        bool got = true;
        if (lane < n_here) got = wait_bar(bar(Lay::bEmpty + slot), ((t_i / KST) & 1u) ^ 1u, abort_flag, err);
        if (!__all_sync(0xffffffffu, got)) {
          aborted = true;
          break;
        }
#ifdef UQ_TEST_STUCK_TILE
        // Test builds only: the first tile of work unit 0 is announced to its
        // barrier but never copied, so that barrier's phase cannot complete
        // and the bounded waits on it run out.  No copy is in flight for that
        // stage.
        const bool copy = !(u == 0 && j0 + lane == 0);
#else
        constexpr bool copy = true;
#endif
        if (lane < n_here) {
          const int tile = U.p_begin + j0 + lane;
          const bool ok = (unsigned)pid < (unsigned)num_blocks;
          reinterpret_cast<volatile int*>(smem + Lay::kSnvOff)[slot] = ok ? min(kPage, U.L - tile * kPage) : 0;
          if (ok) {
            // the stage's previous contents were only read (generic proxy),
            // and the empty barrier orders those reads before this copy
            mbar_arrive_expect_tx(bar(Lay::bFull + slot), kTileBytes);
            if (copy)
              tma_load_3d(stage(slot), &kv_map, 0, U.g, ((pid << lg) + (tile & tmask)) * kPage, bar(Lay::bFull + slot));
          } else {
            atomicOr(err, kErrBadPage);
            mbar_arrive(bar(Lay::bFull + slot));
          }
        }
        tc += (uint32_t)n_here;
      }
      if (aborted) break;
    }
    // copies still in flight (only after an abort): the most recent one of each slot
    const uint32_t n = tc < (uint32_t)KST ? tc : (uint32_t)KST;
    for (uint32_t k = 0; k < n; ++k) {
      const uint32_t t = tc - 1 - k;
      (void)mbar_wait(bar(Lay::bFull + t % KST), (t / KST) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------- tensor core
    // The whole warp walks the schedule and takes every wait; lane 0 issues
    // the tensor-core instructions and their commits.
    // QK: A = K codes E2M1 (format 5), B = q' E4M3 (format 0), UE8M0 scales,
    // N = NR, M = 128; the scale byte of each operand is picked per block.
    const uint32_t idesc_qk = (5u << 7) | ((uint32_t)(NR >> 3) << 17) | (1u << 23) |
                              ((uint32_t)(kGroupTokens >> 4) << 24);
    // PV: D fp32, A and B f16, B (P^T) stored rows-contiguous (MN-major),
    // N = NR, M = 128 head dims.
    const uint32_t idesc_pv = (1u << 4) | (1u << 16) | ((uint32_t)(NR >> 3) << 17) | (8u << 24);
    int un = 0;
    uint32_t gc = 0;
    uint32_t last_bar = 0, last_parity = 0;
    bool issued = false;
    for (;;) {
      const int us = un & 3;
      if (!wait_warp(bar(Lay::bUFull + us), (un >> 2) & 1, abort_flag, err)) break;
      const int u = s_unit[us];
      if (u < 0) break;
      const Unit U = decode_unit(rows, ws, u);
      if (!wait_warp(bar(Lay::bQFull), un & 1, abort_flag, err)) break;
      // Event driven: QK of the next group goes out as soon as its operands
      // are converted and its score buffer is free, PV of the oldest scored
      // group as soon as its P tile is written, whichever comes first.
      bool aborted = false;
      int qk = 0, pv = 0;
      uint32_t idle = 0;
      while (pv < U.n_groups) {
        bool moved = false;
        if (qk < U.n_groups) {
          const uint32_t cg = gc + qk, buf = cg & 1u, sb = cg % NS;
          if (test_warp(bar(Lay::bConv + buf), (cg >> 1) & 1u) &&
              test_warp(bar(Lay::bSFree + sb), ((cg / NS) & 1u) ^ 1u)) {
            tc_fence_after_sync();
            if (lane == 0) {
              const uint32_t ka = sbase + Lay::kKaOff + buf * kKaBytes, qb = sbase + Lay::kQbOff;
#pragma unroll
              for (int kb = 0; kb < 8; ++kb) {
                const uint64_t ad = smem_desc(ka + kb * 2 * kKaChunk, kKaChunk, 128);
                const uint64_t bd = smem_desc(qb + kb * 2 * Lay::kQbChunk, Lay::kQbChunk, 128);
                const uint32_t id = idesc_qk | ((uint32_t)(kb & 3) << 29) | ((uint32_t)(kb & 3) << 4);
                tc_mma_block_scaled(tmem + Lay::kTmS + sb * NR, ad, bd, id,
                                    tmem + Lay::kTmSfa + 8 * buf + 4 * (kb >> 2), tmem + Lay::kTmSfb + 4 * (kb >> 2),
                                    kb > 0 ? 1u : 0u);
              }
              tc_commit(bar(Lay::bSFull + sb));
              tc_commit(bar(Lay::bKaFree + buf));
            }
            __syncwarp();
            last_bar = bar(Lay::bKaFree + buf);
            last_parity = (cg >> 1) & 1u;
            issued = true;
            ++qk;
            moved = true;
          }
        }
        if (pv < qk) {
          const uint32_t pg = gc + pv, buf = pg & 1u;
          if (test_warp(bar(Lay::bPFull + buf), (pg >> 1) & 1u)) {
            tc_fence_after_sync();
            if (lane == 0) {
              const uint32_t pb = sbase + Lay::kPbOff + buf * Lay::kPbBytes;
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                  tc_mma_f16_tmem_a(tmem + Lay::kTmO + h * NR, tmem + Lay::kTmVt + 64 * (2 * buf + h) + 8 * ks,
                                    smem_desc(pb + ks * 256, 128, kPbNGroup), idesc_pv,
                                    (pv > 0 || ks > 0) ? 1u : 0u);
              tc_commit(bar(Lay::bPvDone + buf));
            }
            __syncwarp();
            last_bar = bar(Lay::bPvDone + buf);
            last_parity = (pg >> 1) & 1u;
            ++pv;
            moved = true;
          }
        }
        if (moved) {
          idle = 0;
          continue;
        }
        // nothing ready: sleep on the oldest outstanding event (woken early
        // when it completes), bounded like every other wait
        if (*abort_flag || ++idle > kPollLimit) {
          if (idle > kPollLimit) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeout);
          }
          aborted = true;
          break;
        }
        if (pv < qk) {
          const uint32_t pg = gc + pv;
          poll_bar(bar(Lay::bPFull + (pg & 1u)), (pg >> 1) & 1u);
        } else {
          const uint32_t cg = gc + qk;
          poll_bar(bar(Lay::bConv + (cg & 1u)), (cg >> 1) & 1u);
        }
      }
      if (aborted) break;
      gc += (uint32_t)U.n_groups;
      if (lane == 0) mbar_arrive(bar(Lay::bUEmpty + us));
      ++un;
    }
    // all tensor-core work this warp issued has completed before the CTA ends
    if (issued) (void)mbar_wait(last_bar, last_parity);
  } else if (warp < kSoftWarp0) {
    // ------------------------------------------------------------------ convert
    // A group at a time: wait for its tiles, then the scale metadata of all
    // 128 tokens (four tokens per lane), then the eight tiles as straight-line
    // code whose loads and conversions the scheduler can overlap, then the
    // release of the tiles' stage buffers.
    const int cq = warp & 3;                 // lane quarter: K tiles 2cq, 2cq+1; V dims 64cq ..
    // Shared memory through ordinary loads and stores (addresses in the
    // shared window), which the compiler may batch and reorder; the mbarrier
    // waits and __syncwarp order them where it matters.
    auto ld32 = [&](uint32_t a) { return *reinterpret_cast<const uint32_t*>(smem + (a - sbase)); };
    auto ld64 = [&](uint32_t a) { return *reinterpret_cast<const uint2*>(smem + (a - sbase)); };
    auto ld128 = [&](uint32_t a) { return *reinterpret_cast<const uint4*>(smem + (a - sbase)); };
    auto st32 = [&](uint32_t a, uint32_t v) { *reinterpret_cast<uint32_t*>(smem + (a - sbase)) = v; };
    auto st128 = [&](uint32_t a, uint4 v) { *reinterpret_cast<uint4*>(smem + (a - sbase)) = v; };
    const int gq = lane >> 2, c = lane & 3;
    const uint32_t meta = sbase + Lay::kMetaOff + cq * (kGroupTokens * 4);
    const uint32_t lane_q = (uint32_t)(32 * cq) << 16;
    const uint32_t voff = kVCodeOff + 32 * cq + 4 * gq;
    const uint32_t half_sel = gq < 4 ? 0x5410u : 0x7632u;   // factor of block 2cq or 2cq+1
    const uint32_t vsh = 16u * (cq & 1);                     // blocks 2cq, 2cq+1 in their scale word
    int un = 0;
    uint32_t tc = 0, gc = 0;
    bool aborted = false;
    for (;;) {
      const int us = un & 3;
      if (!wait_warp(bar(Lay::bUFull + us), (un >> 2) & 1, abort_flag, err)) break;
      const int u = s_unit[us];
      if (u < 0) break;
      const Unit U = decode_unit(rows, ws, u);
      for (int grp = 0; grp < U.n_groups; ++grp) {
        const uint32_t buf = gc & 1u, ph = (gc >> 1) & 1u;
        const int n_here = min(kGroupTiles, U.n_tiles - grp * kGroupTiles);
        if (!wait_warp(bar(Lay::bKaFree + buf), ph ^ 1u, abort_flag, err) ||
            !wait_warp(bar(Lay::bPvDone + buf), ph ^ 1u, abort_flag, err)) {
          aborted = true;
          break;
        }
        int nv[kGroupTiles];
        uint32_t sb[kGroupTiles];
#pragma unroll
        for (int i = 0; i < kGroupTiles; ++i) {
          const uint32_t t_i = tc + (uint32_t)i, slot = t_i % KST;
          sb[i] = stage(slot);
          nv[i] = 0;
          if (i < n_here) {
            if (!wait_warp(bar(Lay::bFull + slot), (t_i / KST) & 1u, abort_flag, err)) aborted = true;
            nv[i] = reinterpret_cast<volatile int*>(smem + Lay::kSnvOff)[slot];
          }
        }
        if (aborted) break;
        tc_fence_after_sync();
        // token k = 32 m + lane (tile 2m + lane/16): its largest V block byte
        // E, the relative scales of blocks 2cq and 2cq+1, and (for this
        // quarter's own tokens, m == cq) the V exponent and the K scale bytes
        uint32_t sfw0 = 0, sfw1 = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const bool hi = lane >= 16;
          const int nvt = hi ? nv[2 * m + 1] : nv[2 * m];
          const uint32_t row = (hi ? sb[2 * m + 1] : sb[2 * m]) + (lane & 15) * kSlotBytes;
          uint32_t f = 0u, E = 0u;
          if (nvt > 0) {
            const uint2 sc = ld64(row + kVScaleOff);
            E = max_byte8(sc.x, sc.y);
            const uint32_t w = cq < 2 ? sc.x : sc.y;
            f = pow2_rel_f16x2((E - ((w >> vsh) & 0xffu)) | ((E - ((w >> (vsh + 8)) & 0xffu)) << 16));
            if (m == cq) {
              const uint2 ks = ld64(row + kKScaleOff);
              sfw0 = ks.x;
              sfw1 = ks.y;
            }
          }
          st32(meta + 4 * (32 * m + lane), f);
          if (m == cq)
            st32(sbase + Lay::kEvfOff + (buf * kGroupTokens + 32 * m + lane) * 4,
                  __float_as_uint(nvt > 0 ? (float)((int)E - 127 - kRelTop) : 0.f));
        }
#pragma unroll
        for (int i = 0; i < kGroupTiles; ++i)
          if ((i >> 1) == cq && lane == (i & 1)) st32(sbase + Lay::kGnvOff + (buf * kGroupTiles + i) * 4, (uint32_t)nv[i]);
        __syncwarp();
        // V: tokens 2c, 2c+1 (pair A) and 2c+8, 2c+9 (pair B) of each tile,
        // head dims 64cq + 8gq .. +7; the same dim of a pair shares one byte
#pragma unroll
        for (int i = 0; i < kGroupTiles; ++i) {
          const uint32_t vt = tmem + lane_q + Lay::kTmVt + 64 * (2 * buf) + 8 * i;
          uint32_t LA[4] = {0u, 0u, 0u, 0u}, HA[4] = {0u, 0u, 0u, 0u}, LB[4] = {0u, 0u, 0u, 0u},
                   HB[4] = {0u, 0u, 0u, 0u};
          if (nv[i] > 0) {
            const uint32_t x0 = ld32(sb[i] + (2 * c) * kSlotBytes + voff);
            const uint32_t x1 = ld32(sb[i] + (2 * c + 1) * kSlotBytes + voff);
            const uint32_t x2 = ld32(sb[i] + (2 * c + 8) * kSlotBytes + voff);
            const uint32_t x3 = ld32(sb[i] + (2 * c + 9) * kSlotBytes + voff);
            const uint32_t mt = meta + 4 * (16 * i + 2 * c);
            const uint32_t rvA = __byte_perm(ld32(mt), ld32(mt + 4), half_sel);
            const uint32_t rvB = __byte_perm(ld32(mt + 32), ld32(mt + 36), half_sel);
            f16x2x4_from_e2m1_word((x0 & 0x0F0F0F0Fu) | ((x1 << 4) & 0xF0F0F0F0u), LA);
            f16x2x4_from_e2m1_word(((x0 >> 4) & 0x0F0F0F0Fu) | (x1 & 0xF0F0F0F0u), HA);
            f16x2x4_from_e2m1_word((x2 & 0x0F0F0F0Fu) | ((x3 << 4) & 0xF0F0F0F0u), LB);
            f16x2x4_from_e2m1_word(((x2 >> 4) & 0x0F0F0F0Fu) | (x3 & 0xF0F0F0F0u), HB);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              LA[e] = hmul2(LA[e], rvA);
              HA[e] = hmul2(HA[e], rvA);
              LB[e] = hmul2(LB[e], rvB);
              HB[e] = hmul2(HB[e], rvB);
            }
          }
          // half h, m-tile mt: dims 8gq + 4h + 2mt (+1) at lanes 16mt + gq (+8);
          // a missing or rejected tile leaves finite zeros
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
              tmem_st_16x128b_x2(vt + ((uint32_t)(16 * mt) << 16) + 64 * h, LA[2 * h + mt], HA[2 * h + mt],
                                 LB[2 * h + mt], HB[2 * h + mt]);
        }
        // K codes of this quarter's tiles 2cq, 2cq+1 into rows 32cq .. 32cq+31
        // of the K operand (16-element chunks of 8 code bytes and 8 unused)
        const uint32_t ka = sbase + Lay::kKaOff + buf * kKaBytes;
#pragma unroll
        for (int i = 0; i < kGroupTiles; ++i) {
          if ((i >> 1) == cq && nv[i] > 0) {
            // all four loads before any store: the stores could alias them
            // as far as the compiler knows
            uint4 v[4];
#pragma unroll
            for (int rep = 0; rep < 4; ++rep) {
              const int idx = rep * 32 + lane, t = idx & 15, m = idx >> 4;   // token fastest
              v[rep] = ld128(sb[i] + t * kSlotBytes + 16 * m);
            }
#pragma unroll
            for (int rep = 0; rep < 4; ++rep) {
              const int idx = rep * 32 + lane, t = idx & 15, m = idx >> 4;
              const int row = 16 * i + t;
              const uint32_t base = ka + (row >> 3) * 128 + (row & 7) * 16;
              st128(base + (2 * m) * kKaChunk, make_uint4(v[rep].x, v[rep].y, 0u, 0u));
              st128(base + (2 * m + 1) * kKaChunk, make_uint4(v[rep].z, v[rep].w, 0u, 0u));
            }
          }
        }
        // K scales of the quarter's 32 token lanes: blocks 0-3 in column +0,
        // blocks 4-7 in column +4 (one byte per block)
        const uint32_t sfv[8] = {sfw0, sfw0, sfw0, sfw0, sfw1, sfw1, sfw1, sfw1};
        tmem_st_32x32b_x8(tmem + lane_q + Lay::kTmSfa + 8 * buf, sfv);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(Lay::bConv + buf));
#pragma unroll
          for (int i = 0; i < kGroupTiles; ++i)
            if (i < n_here) mbar_arrive(bar(Lay::bEmpty + (tc + (uint32_t)i) % KST));
        }
        tc += (uint32_t)n_here;
        ++gc;
      }
      if (aborted) break;
      if (lane == 0) mbar_arrive(bar(Lay::bUEmpty + us));
      ++un;
    }
  } else {
    // ------------------------------------------------------------------ softmax
    const int sq = warp & 3;                  // lane quarter: tokens 32sq .. of a group; O^T dims
    const int sw = warp - kSoftWarp0;         // 0..3
    const int st = threadIdx.x - kSoftWarp0 * 32;
    const uint32_t lane_q = (uint32_t)(32 * sq) << 16;
    float* s_m = reinterpret_cast<float*>(smem + Lay::kStatOff);
    float* s_d = s_m + NR;
    int* s_rlo = reinterpret_cast<int*>(smem + Lay::kRowOff);
    int* s_rhi = s_rlo + NR;
    float* red = reinterpret_cast<float*>(smem + Lay::kRedOff);   // [4][2][NR]
    float* fac = reinterpret_cast<float*>(smem + Lay::kFacOff);
    // q' carries no block scales: 2^0 in every scale byte
    {
      const uint32_t ones[8] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
                                0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
      tmem_st_32x32b_x8(tmem + lane_q + Lay::kTmSfb, ones);
      tmem_wait_st();
      tc_fence_before_sync();
    }
    int un = 0;
    uint32_t gc = 0;
    for (;;) {
      const int us = un & 3;
      const bool got = wait_warp(bar(Lay::bUFull + us), (un >> 2) & 1, abort_flag, err);
      if (bar_or_named(kSoftBar, kSoftThreads, !got)) break;
      const int u = s_unit[us];
      if (u < 0) break;
      const Unit U = decode_unit(rows, ws, u);
      const int pack = rows.pack;
      const int last_row = unit_last_row(rows, U.b);
      auto row_pos = [&](int r) { return U.b * pack + r / QG; };
      auto row_exists = [&](int r) { return r < QG * pack && row_pos(r) <= last_row; };
      // ---- unit prologue: row ranges, running state, q' in operand layout
      if (st < NR) {
        const int r = st;
        int lo = 0x7fffffff, hi = -1;
        if (row_exists(r)) {
          hi = row_len(rows, row_pos(r));
          lo = row_lo(rows, hi);
        }
        s_rlo[r] = lo;
        s_rhi[r] = hi;
        s_m[r] = -INFINITY;
        s_d[r] = -INFINITY;
      }
      for (int r = sw; r < NR; r += 4) {
        uint32_t w0 = 0u, w1 = 0u;
        if (row_exists(r)) {
          const uint16_t* qp = query + (int64_t)row_pos(r) * q_ss + (int64_t)(U.g * QG + r % QG) * q_sh + lane * 8;
          const uint4 raw = *reinterpret_cast<const uint4*>(qp);
          float x[8];
          const uint32_t uu[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            x[2 * i] = bf16_bits_to_f32(uu[i] & 0xffffu);
            x[2 * i + 1] = bf16_bits_to_f32(uu[i] >> 16);
          }
          // the fast Walsh-Hadamard butterfly in its canonical stage order:
          // strides 1, 2, 4 in registers, 8 .. 128 across lanes
#pragma unroll
          for (int hh = 1; hh < 8; hh <<= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if ((i & hh) == 0) {
                const float a = x[i], b2 = x[i + hh];
                x[i] = a + b2;
                x[i + hh] = a - b2;
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
          w0 = e4m3x4_from_f32(x[0] * 0.0625f, x[1] * 0.0625f, x[2] * 0.0625f, x[3] * 0.0625f);
          w1 = e4m3x4_from_f32(x[4] * 0.0625f, x[5] * 0.0625f, x[6] * 0.0625f, x[7] * 0.0625f);
        }
        // head dims 8 lane .. 8 lane + 7: chunk lane / 2, bytes 8 (lane % 2) ..
        sts64(sbase + Lay::kQbOff + (lane >> 1) * Lay::kQbChunk + (r >> 3) * 128 + (r & 7) * 16 + 8 * (lane & 1),
              w0, w1);
      }
      fence_proxy_async_smem();
      bar_sync_named(kSoftBar, kSoftThreads);
      if (lane == 0) mbar_arrive(bar(Lay::bQFull));
      // the group range inside which no row needs its own mask
      int full_lo = 0, full_hi = 0x7fffffff;
      for (int r = 0; r < NR; ++r)
        if (s_rhi[r] >= 0) {
          full_lo = max(full_lo, s_rlo[r]);
          full_hi = min(full_hi, s_rhi[r]);
        }
      float lp[NR];   // this token lane's share of each row's sum of 2^(s - m)
#pragma unroll
      for (int r = 0; r < NR; ++r) lp[r] = 0.f;
      const int t = 32 * sq + lane;           // token of the group
      bool aborted = false;
      for (int grp = 0; grp < U.n_groups; ++grp) {
        const uint32_t cg = gc + grp, buf = cg & 1u, sb = cg % NS;
        bool ok = wait_warp(bar(Lay::bSFull + sb), (cg / NS) & 1u, abort_flag, err);
        ok = ok && wait_warp(bar(Lay::bConv + buf), (cg >> 1) & 1u, abort_flag, err);
        ok = ok && wait_warp(bar(Lay::bPvDone + buf), ((cg >> 1) & 1u) ^ 1u, abort_flag, err);
        if (bar_or_named(kSoftBar, kSoftThreads, !ok)) {
          aborted = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t s_col = tmem + lane_q + Lay::kTmS + sb * NR;
        const int tile = t >> 4;
        const int nv = reinterpret_cast<const int*>(smem + Lay::kGnvOff)[buf * kGroupTiles + tile];
        const bool tok_ok = (t & 15) < nv;
        const int g0 = (U.p_begin + grp * kGroupTiles) * kPage;
        const int t_abs = g0 + t;
        const float ev = reinterpret_cast<const float*>(smem + Lay::kEvfOff)[buf * kGroupTokens + t];
        const bool masks = g0 < full_lo || g0 + kGroupTokens > full_hi;
        const uint32_t pb = sbase + Lay::kPbOff + buf * Lay::kPbBytes + t * 16;
        // rows in chunks of up to 32: one tensor-memory load each, the scores
        // then stay in registers for the vote, the rare update and the weights
#pragma unroll
        for (int c0 = 0; c0 < NR; c0 += kChunk) {
          float sv[kChunk];
          tmem_ld_cols(s_col + c0, sv);
#pragma unroll
          for (int k = 0; k < kChunk; ++k) {
            bool okk = tok_ok;
            if (masks) okk = okk && t_abs >= s_rlo[c0 + k] && t_abs < s_rhi[c0 + k];
            sv[k] = okk ? sv[k] * scale_log2e : -INFINITY;
          }
          bool grow = false;
#pragma unroll
          for (int r0 = 0; r0 < kChunk; r0 += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(s_m + c0 + r0);
            const float4 d4 = *reinterpret_cast<const float4*>(s_d + c0 + r0);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float sc = sv[r0 + k];
              const float m_ref = mm[k] == -INFINITY ? 0.f : mm[k];
              grow |= sc > mm[k] + kLazyMaxLog2;
              grow |= (sc - m_ref) + ev > dd[k] + kLazyMaxLog2;
            }
          }
          if (bar_or_named(kSoftBar, kSoftThreads, grow)) {
            // rare: new running maxima for the chunk's rows.  1) the group's
            // row maxima of s
#pragma unroll
            for (int k = 0; k < kChunk; ++k) {
              float x = sv[k];
#pragma unroll
              for (int msk = 1; msk < 32; msk <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, msk));
              if (lane == 0) red[(sq * 2) * NR + c0 + k] = x;
            }
            bar_sync_named(kSoftBar, kSoftThreads);
            // 2) the new m, and the maxima of the V exponents relative to it
#pragma unroll
            for (int k = 0; k < kChunk; ++k) {
              const int r = c0 + k;
              const float tm = fmaxf(fmaxf(red[0 * NR + r], red[2 * NR + r]), fmaxf(red[4 * NR + r], red[6 * NR + r]));
              const float m_old = s_m[r];
              const float m_new = tm > m_old + kLazyMaxLog2 ? tm : m_old;
              if (m_new != m_old) lp[r] *= fast_exp2(m_old - m_new);
              const float m_ref = m_new == -INFINITY ? 0.f : m_new;
              float y = (sv[k] - m_ref) + ev;
#pragma unroll
              for (int msk = 1; msk < 32; msk <<= 1) y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, msk));
              if (lane == 0) red[(sq * 2 + 1) * NR + r] = y;
            }
            bar_sync_named(kSoftBar, kSoftThreads);
            // 3) one thread per row moves the state; fac = O's factor
            bool moved = false;
            if (st < kChunk) {
              const int r = c0 + st;
              const float tm = fmaxf(fmaxf(red[0 * NR + r], red[2 * NR + r]), fmaxf(red[4 * NR + r], red[6 * NR + r]));
              const float ym = fmaxf(fmaxf(red[1 * NR + r], red[3 * NR + r]), fmaxf(red[5 * NR + r], red[7 * NR + r]));
              const float m_old = s_m[r], d_old = s_d[r];
              const float m_new = tm > m_old + kLazyMaxLog2 ? tm : m_old;
              const float d_cur = m_old == -INFINITY ? -INFINITY : d_old + (m_old - m_new);
              const float d_new = ym > d_cur + kLazyMaxLog2 ? ym : d_cur;
              fac[r] = d_new == d_cur ? 1.f : fast_exp2(d_cur - d_new);
              moved = d_new != d_cur;
              s_m[r] = m_new;
              s_d[r] = d_new;
            }
            const bool resc = bar_or_named(kSoftBar, kSoftThreads, moved);   // also publishes s_m, s_d, fac
            if (resc && grp > 0) {
              // O^T holds the groups so far: wait for the last one's PV, then
              // scale the chunk rows' columns by their factors
              const uint32_t pg = cg - 1;
              const bool okr = wait_warp(bar(Lay::bPvDone + (pg & 1u)), (pg >> 1) & 1u, abort_flag, err);
              if (bar_or_named(kSoftBar, kSoftThreads, !okr)) {
                aborted = true;
                break;
              }
              tc_fence_after_sync();
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int r0 = 0; r0 < kChunk; r0 += 16) {
                  float o[16];
                  tmem_ld16(tmem + lane_q + Lay::kTmO + h * NR + c0 + r0, o);
#pragma unroll
                  for (int k = 0; k < 16; ++k) o[k] *= fac[c0 + r0 + k];
                  tmem_st16(tmem + lane_q + Lay::kTmO + h * NR + c0 + r0, o);
                }
              tmem_wait_st();
            }
          }
          // probabilities: l and the f16 PV weights, P^T rows-contiguous per token
#pragma unroll
          for (int r8 = 0; r8 < kChunk; r8 += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int r0 = r8 + 4 * half;
              const float4 m4 = *reinterpret_cast<const float4*>(s_m + c0 + r0);
              const float4 d4 = *reinterpret_cast<const float4*>(s_d + c0 + r0);
              const float mm[4] = {m4.x, m4.y, m4.z, m4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
              float wv[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float m_ref = mm[k] == -INFINITY ? 0.f : mm[k];
                const float d_ref = dd[k] == -INFINITY ? 0.f : dd[k];
                const float x = sv[r0 + k] - m_ref;
                lp[c0 + r0 + k] += fast_exp2(x);
                wv[k] = fast_exp2((x + ev) - d_ref);
              }
              pk[2 * half] = pack_f16x2(wv[0], wv[1]);
              pk[2 * half + 1] = pack_f16x2(wv[2], wv[3]);
            }
            sts128(pb + ((c0 + r8) >> 3) * kPbNGroup, make_uint4(pk[0], pk[1], pk[2], pk[3]));
          }
        }
        if (aborted) break;
        tc_fence_before_sync();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(Lay::bSFree + sb));
          mbar_arrive(bar(Lay::bPFull + buf));
        }
      }
      if (aborted) break;
      gc += (uint32_t)U.n_groups;
      // ---- unit end: the last PV, the row sums, the split partial
      bool ok = true;
      if (U.n_groups > 0) ok = wait_warp(bar(Lay::bPvDone + ((gc - 1) & 1u)), ((gc - 1) >> 1) & 1u, abort_flag, err);
      if (bar_or_named(kSoftBar, kSoftThreads, !ok)) break;
      tc_fence_after_sync();
      // lane r of each warp gets the warp's sum of row r (32 rows per pass)
#pragma unroll
      for (int r0 = 0; r0 < NR; r0 += 32) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (r0 + j < NR) ? lp[r0 + j] : 0.f;
#pragma unroll
        for (int k = 16; k >= 1; k >>= 1)
#pragma unroll
          for (int j = 0; j < k; ++j) {
            const float send = (lane & k) ? v[j] : v[j + k];
            const float keep = (lane & k) ? v[j + k] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, k);
          }
        if (r0 + lane < NR) red[(sq * 2) * NR + r0 + lane] = v[0];
      }
      bar_sync_named(kSoftBar, kSoftThreads);
      if (st < NR) {
        const int r = st;
        const float L = red[0 * NR + r] + red[2 * NR + r] + red[4 * NR + r] + red[6 * NR + r];
        fac[r] = L > 0.f ? fast_exp2(s_d[r]) / L : 0.f;
        if (row_exists(r)) {
          const int64_t orow = (int64_t)row_pos(r) * Hq + U.g * QG + r % QG;
          ws.part_lse[orow * S + U.split] = L > 0.f ? s_m[r] + fast_log2(L) : -INFINITY;
        }
      }
      bar_sync_named(kSoftBar, kSoftThreads);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int dim = lane_dim(sq, h, lane);
#pragma unroll
        for (int r0 = 0; r0 < NR; r0 += 16) {
          float o[16];
          tmem_ld16(tmem + lane_q + Lay::kTmO + h * NR + r0, o);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int r = r0 + k;
            if (row_exists(r)) {
              const int64_t orow = (int64_t)row_pos(r) * Hq + U.g * QG + r % QG;
              ws.part_o[(orow * S + U.split) * kHeadDim + dim] = o[k] * fac[r];
            }
          }
        }
      }
      tc_fence_before_sync();
      bar_sync_named(kSoftBar, kSoftThreads);   // fac and red are free for the next unit
      if (st == 0) misc[2] = un + 1;             // units whose partials are written
      if (lane == 0) mbar_arrive(bar(Lay::bUEmpty + us));
      ++un;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (warp == kProducerWarp && *abort_flag) {
    // After an abort, the units this CTA took but did not finish get empty
    // split partials (log-sum-exp -inf, output 0), so that the merge skips
    // them: the rows lose those splits instead of reading stale partials.
    for (int k = misc[2]; k <= published; ++k) {
      const int u = k < published ? s_unit[k & 3] : pending;
      if (u < 0) continue;
      const Unit U = decode_unit(rows, ws, u);
      const int pack = rows.pack, last_row = unit_last_row(rows, U.b);
      for (int r = 0; r < QG * pack; ++r) {
        const int pos = U.b * pack + r / QG;
        if (pos > last_row) break;
        const int64_t idx = ((int64_t)pos * Hq + U.g * QG + r % QG) * S + U.split;
        if (lane == 0) ws.part_lse[idx] = -INFINITY;
        for (int d = lane; d < kHeadDim; d += 32) ws.part_o[idx * kHeadDim + d] = 0.f;
      }
    }
  }
}

}  // namespace wide

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
cudaError_t current_context_id(unsigned long long* id);
cudaError_t make_kv_tensor_map(CUtensorMap* map, const uint8_t* kv, int Hk, int64_t num_slots);

// Rows of a wide unit for a launch: 16, 32 or 64 (the kernel's N).
int wide_rows(int rows_per_unit) { return rows_per_unit <= 16 ? 16 : rows_per_unit <= 32 ? 32 : 64; }

static std::mutex g_wide_mutex;

template <int NR>
static cudaError_t wide_grid(int* grid) {
  using Lay = wide::Layout<NR>;
  static int grid_of_device[64] = {0};
  static unsigned long long ctx_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned long long ctx = 0;
  if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_wide_mutex);
  if (dev >= 0 && dev < 64 && grid_of_device[dev] > 0 && ctx_of_device[dev] == ctx) {
    *grid = grid_of_device[dev];
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(wide::decode_stage1_wide<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  *grid = sms;   // one CTA per SM: it holds all 512 tensor-memory columns
  if (dev >= 0 && dev < 64) {
    grid_of_device[dev] = *grid;
    ctx_of_device[dev] = ctx;
  }
  return cudaSuccess;
}

cudaError_t launch_wide_stage1(int rows_per_unit, const uint16_t* query, int64_t q_ss, int64_t q_sh,
                               const CUtensorMap& kv_map, const int32_t* bt, const SeqRows& sl, float scale,
                               int Hq, int Hk, int num_blocks, int S, const Workspace& ws, unsigned* err,
                               cudaStream_t stream, int grid);

template <int NR>
static cudaError_t launch_wide_nr(const uint16_t* query, int64_t q_ss, int64_t q_sh, const CUtensorMap& kv_map,
                                  const int32_t* bt, const SeqRows& sl, float scale, int Hq, int Hk,
                                  int num_blocks, int S, const Workspace& ws, unsigned* err,
                                  cudaStream_t stream, int grid) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(wide::kThreads);
  cfg.dynamicSmemBytes = wide::Layout<NR>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wide::decode_stage1_wide<NR>, query, q_ss, q_sh, kv_map, bt, sl,
                            scale * kLog2e, Hq, Hk, num_blocks, S, ws, err);
}

cudaError_t wide_stage1_grid(int rows_per_unit, int* grid) {
  switch (wide_rows(rows_per_unit)) {
    case 16: return wide_grid<16>(grid);
    case 32: return wide_grid<32>(grid);
    default: return wide_grid<64>(grid);
  }
}

cudaError_t launch_wide_stage1(int rows_per_unit, const uint16_t* query, int64_t q_ss, int64_t q_sh,
                               const CUtensorMap& kv_map, const int32_t* bt, const SeqRows& sl, float scale,
                               int Hq, int Hk, int num_blocks, int S, const Workspace& ws, unsigned* err,
                               cudaStream_t stream, int grid) {
  switch (wide_rows(rows_per_unit)) {
    case 16:
      return launch_wide_nr<16>(query, q_ss, q_sh, kv_map, bt, sl, scale, Hq, Hk, num_blocks, S, ws, err, stream, grid);
    case 32:
      return launch_wide_nr<32>(query, q_ss, q_sh, kv_map, bt, sl, scale, Hq, Hk, num_blocks, S, ws, err, stream, grid);
    default:
      return launch_wide_nr<64>(query, q_ss, q_sh, kv_map, bt, sl, scale, Hq, Hk, num_blocks, S, ws, err, stream, grid);
  }
}

}  // namespace uq
