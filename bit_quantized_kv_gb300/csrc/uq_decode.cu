// uq_decode.cu -- split-KV paged decode attention over the FP4 E2M1 + UE8M0
// cache (vllm.v1.attention.ops.flydsl_ultraquant_decode,
// flydsl_ultraquant_decode_attention: query prologue with the E4M3 haircut,
// stage-1 split partials, partition reduce; the fixed split count follows
// vllm.v1.attention.ops.turboquant_soa.triton_turboquant_decode_v2).
//
// Stage 1: one CTA per (split, kv head, sequence), 4 warps.  A split is a run
// of whole 16-token pages; each warp takes every 4th page of it and keeps its
// own online-softmax state.  A page's 16 slots of one kv head (16 x 272 B)
// are brought into shared memory by bulk async copies that complete on a
// per-stage mbarrier, NSTAGE pages ahead.  The CTA's query group (6, 8 or 16
// rows) is rotated once (fp32 butterfly, x 1/16), rounded through E4M3, and
// kept as f16 tensor-core fragments.
//
// Tensor-core formulation (mma.m16n8k16, f16 in, fp32 accumulate):
//   QK:  S[t, r] = sum_d K'[t, d] Q'[r, d]      (M = 16 tokens, N = 8 rows)
//   PV:  O^T[d, r] += sum_t V'[t, d] W[r, t]    (M = 16 head dims, N = 8 rows)
// Every FP4 value is c * 2^(e_blk - 127).  For each token t the largest
// block exponent E_t is factored out, so K' = c * 2^(e_blk - E_t) and
// V' = c * 2^(e_blk - E_t) are exact in f16 whenever e_blk >= E_t - 23 (a
// block more than 2^23 below the token's largest block contributes below
// f16's range and is dropped).  2^(E^K_t - 127) multiplies the scores;
// 2^(E^V_t - 127) is added to the exponent of the probability that weights
// the token's V' row.  The contraction index of QK may be permuted freely as
// long as Q' and K' agree, which lets every lane read contiguous bytes:
// lane (g = lane/4, c = lane%4) owns head dims [64c, 64c+64) of K (k-step i
// covers 64c + 4i .. +3) and V head dims [32g, 32g+32) (one UE8M0 block).
//
// Stage 2: one warp per (sequence, query head) merges the active splits with
// the log-sum-exp rule and writes bf16.
#include "uq_device.cuh"

namespace uq {

constexpr int kPage = 16;                        // tokens per page (block_size)
constexpr int kTileBytes = kPage * kSlotBytes;   // 4352 bytes per (page, kv head)
constexpr int kMinPagesPerSplit = 8;             // floor of 128 tokens per split
constexpr float kLog2e = 1.4426950408889634f;

struct SplitPlan {
  int pages_per_split;
  int n_active;
};

// Split assignment, identical in both stages: up to S splits of whole pages,
// each at least kMinPagesPerSplit pages unless the sequence is shorter.
__device__ __forceinline__ SplitPlan split_plan(int L, int S) {
  const int P = (L + kPage - 1) / kPage;
  if (P <= 0) return {0, 0};
  const int want = (P + kMinPagesPerSplit - 1) / kMinPagesPerSplit;
  const int ns = min(S, max(1, want));
  const int pps = (P + ns - 1) / ns;
  return {pps, (P + pps - 1) / pps};
}

__device__ __forceinline__ int clamp_len(int L, int max_blocks) {
  L = max(L, 0);
  const long long cap = (long long)max_blocks * kPage;
  return (long long)L > cap ? (int)cap : L;
}

template <int NT, int NWARPS, int NSTAGE>
struct Stage1Layout {
  static constexpr int kRows = NT * 8;                       // padded query rows
  static constexpr int kStageBytes = NWARPS * NSTAGE * kTileBytes;
  static constexpr int kORowStride = kHeadDim + 4;           // floats
  static constexpr int kMergeBytes = NWARPS * kRows * kORowStride * 4;
  static constexpr int kUnionBytes = kStageBytes > kMergeBytes ? kStageBytes : kMergeBytes;
  static constexpr int kStatsOff = kUnionBytes;              // [NWARPS][kRows][4] floats
  static constexpr int kStatsBytes = NWARPS * kRows * 4 * 4;
  static constexpr int kRowInfoOff = kStatsOff + kStatsBytes; // [kRows][NWARPS+2] floats
  static constexpr int kRowInfoBytes = kRows * (NWARPS + 2) * 4;
  static constexpr int kBarOff = (kRowInfoOff + kRowInfoBytes + 15) / 16 * 16;
  static constexpr int kBarBytes = NWARPS * NSTAGE * 8;
  static constexpr int kQOff = (kBarOff + kBarBytes + 127) / 128 * 128;
  static constexpr int kQBytes = kRows * kHeadDim * 2;      // f16 [kRows][256]
  static constexpr int kBytes = kQOff + kQBytes;
};

template <int NT, int NWARPS, int NSTAGE>
__global__ void __launch_bounds__(NWARPS * 32, NT == 1 ? 3 : 2)
decode_stage1(const uint16_t* __restrict__ query, int64_t q_ss, int64_t q_sh,
              const uint8_t* __restrict__ kv, const int32_t* __restrict__ block_table,
              const int32_t* __restrict__ seq_lens, float scale_log2e, int Hq, int Hk,
              int QG, int num_blocks, int max_blocks, int S, float* __restrict__ part_o,
              float* __restrict__ part_lse, unsigned* __restrict__ err) {
  using Lay = Stage1Layout<NT, NWARPS, NSTAGE>;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int L = clamp_len(seq_lens[b], max_blocks);
  const SplitPlan plan = split_plan(L, S);
  if (split >= plan.n_active) return;
  const int P = (L + kPage - 1) / kPage;
  const int p_begin = split * plan.pages_per_split;
  const int p_end = min(p_begin + plan.pages_per_split, P);

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + Lay::kBarOff + warp * NSTAGE * 8;
  const uint32_t stage_base = smem_base + warp * NSTAGE * kTileBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NWARPS * NSTAGE; ++i) mbar_init(smem_base + Lay::kBarOff + 8 * i, 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- per-warp page schedule -------------------------------------------
  const int n_pages = p_end - p_begin;
  const int n_my = n_pages > warp ? (n_pages - warp + NWARPS - 1) / NWARPS : 0;
  const int32_t* bt_row = block_table + (int64_t)b * max_blocks + p_begin + warp;
  int pid_chunk = -1, pid_reg = -1;
  uint32_t stage_ok = 0;  // bit s: stage s holds a page that was really copied

  auto issue = [&](int j) {
    const int chunk = j >> 5;
    if (chunk != pid_chunk) {
      const int jj = chunk * 32 + lane;
      pid_reg = jj < n_my ? bt_row[(int64_t)jj * NWARPS] : -1;
      pid_chunk = chunk;
    }
    const int pid = __shfl_sync(0xffffffffu, pid_reg, j & 31);
    const int stg = j % NSTAGE;
    const uint32_t bar = bar_base + 8 * stg;
    const bool ok = (unsigned)pid < (unsigned)num_blocks;
    stage_ok = ok ? (stage_ok | (1u << stg)) : (stage_ok & ~(1u << stg));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (ok) {
        mbar_arrive_expect_tx(bar, kTileBytes);
      } else {
        atomicOr(err, kErrBadPage);
        mbar_arrive(bar);
      }
    }
    __syncwarp();
    if (ok && lane < kPage) {
      const uint8_t* src = kv + (((int64_t)pid * kPage + lane) * Hk + g) * (int64_t)kSlotBytes;
      bulk_g2s(stage_base + stg * kTileBytes + lane * kSlotBytes, src, kSlotBytes, bar);
    }
  };

  for (int j = 0; j < NSTAGE && j < n_my; ++j) issue(j);

  // ---- query prologue: q' = f16(e4m3(fp32(q) H)) --------------------------
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + Lay::kQOff);
  for (int r = warp; r < Lay::kRows; r += NWARPS) {
    uint4 packed = make_uint4(0, 0, 0, 0);
    if (r < QG) {
      const uint16_t* qp = query + (int64_t)b * q_ss + (int64_t)(g * QG + r) * q_sh + lane * 8;
      const uint4 raw = *reinterpret_cast<const uint4*>(qp);
      float x[8];
      const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_bits_to_f32(u[i] & 0xffffu);
        x[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
      }
#pragma unroll
      for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((i & h) == 0) {
            const float a = x[i], c = x[i + h];
            x[i] = a + c;
            x[i + h] = a - c;
          }
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
          x[i] = upper ? (other - x[i]) : (x[i] + other);
        }
      }
      packed.x = e4m3_roundtrip_f16x2(x[0] * 0.0625f, x[1] * 0.0625f);
      packed.y = e4m3_roundtrip_f16x2(x[2] * 0.0625f, x[3] * 0.0625f);
      packed.z = e4m3_roundtrip_f16x2(x[4] * 0.0625f, x[5] * 0.0625f);
      packed.w = e4m3_roundtrip_f16x2(x[6] * 0.0625f, x[7] * 0.0625f);
    }
    *reinterpret_cast<uint4*>(qs + r * kHeadDim + lane * 8) = packed;
  }
  __syncthreads();

  const int gq = lane >> 2, c = lane & 3;
  // Q' B-fragments: k-step i, lane (gq, c): row 8nt+gq, head dims 64c+4i .. +3
  uint32_t qf[NT][16][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t base = smem_u32(qs + (nt * 8 + gq) * kHeadDim + 64 * c);
#pragma unroll
    for (int i2 = 0; i2 < 8; ++i2) {
      const uint4 v = lds128(base + 16 * i2);
      qf[nt][2 * i2][0] = v.x;
      qf[nt][2 * i2][1] = v.y;
      qf[nt][2 * i2 + 1][0] = v.z;
      qf[nt][2 * i2 + 1][1] = v.w;
    }
  }

  // ---- main loop ------------------------------------------------------------
  float o[NT][16][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
  float m_run[NT][2], mu_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m_run[nt][h] = -INFINITY;
      mu_run[nt][h] = -INFINITY;
      l_run[nt][h] = 0.f;
    }

  const int ta = 2 * c, tb = 2 * c + 1, tcc = 2 * c + 8, td = 2 * c + 9;
  bool timed_out = false;
  int j = 0;
  for (; j < n_my; ++j) {
    const int stg = j % NSTAGE;
    if (!mbar_wait(bar_base + 8 * stg, (uint32_t)((j / NSTAGE) & 1))) {
      timed_out = true;
      break;
    }
    const int page = p_begin + warp + j * NWARPS;
    const int nvalid = ((stage_ok >> stg) & 1u) ? min(kPage, L - page * kPage) : 0;
    if (nvalid > 0) {
      const uint32_t sb = stage_base + stg * kTileBytes;
      // -- K scales of tokens gq, gq+8: token max E and the relative scales of
      //    blocks 2c, 2c+1 as f16x2 (both halves equal)
      const uint2 ks0 = lds64(sb + gq * kSlotBytes + kKScaleOff);
      const uint2 ks1 = lds64(sb + (gq + 8) * kSlotBytes + kKScaleOff);
      const uint32_t ek0 = max_byte8(ks0.x, ks0.y), ek1 = max_byte8(ks1.x, ks1.y);
      const uint32_t kw0 = (c < 2) ? ks0.x : ks0.y, kw1 = (c < 2) ? ks1.x : ks1.y;
      const int sh = 16 * (c & 1);
      uint32_t rk0[2], rk1[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t h0 = pow2_neg_f16((int)ek0 - (int)((kw0 >> (sh + 8 * q)) & 0xffu));
        const uint32_t h1 = pow2_neg_f16((int)ek1 - (int)((kw1 >> (sh + 8 * q)) & 0xffu));
        rk0[q] = h0 | (h0 << 16);
        rk1[q] = h1 | (h1 << 16);
      }
      // -- QK on the tensor cores
      const uint4 ka0 = lds128(sb + gq * kSlotBytes + 32 * c);
      const uint4 ka1 = lds128(sb + gq * kSlotBytes + 32 * c + 16);
      const uint4 kb0 = lds128(sb + (gq + 8) * kSlotBytes + 32 * c);
      const uint4 kb1 = lds128(sb + (gq + 8) * kSlotBytes + 32 * c + 16);
      const uint32_t kaw[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
      const uint32_t kbw[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
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
        for (int half = 0; half < 2; ++half) {
          const int i = 2 * q + half;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16_16816(sacc[nt], fa[2 * half], fb[2 * half], fa[2 * half + 1],
                          fb[2 * half + 1], qf[nt][i][0], qf[nt][i][1]);
        }
      }
      // -- V scales: tokens 2c, 2c+1, 2c+8, 2c+9 (E and block gq byte)
      const uint2 vsa = lds64(sb + ta * kSlotBytes + kVScaleOff);
      const uint2 vsb = lds64(sb + tb * kSlotBytes + kVScaleOff);
      const uint2 vsc = lds64(sb + tcc * kSlotBytes + kVScaleOff);
      const uint2 vsd = lds64(sb + td * kSlotBytes + kVScaleOff);
      const uint32_t eva = max_byte8(vsa.x, vsa.y), evb = max_byte8(vsb.x, vsb.y);
      const uint32_t evc = max_byte8(vsc.x, vsc.y), evd = max_byte8(vsd.x, vsd.y);
      const int bsh = 8 * (gq & 3);
      const uint32_t bya = (((gq < 4) ? vsa.x : vsa.y) >> bsh) & 0xffu;
      const uint32_t byb = (((gq < 4) ? vsb.x : vsb.y) >> bsh) & 0xffu;
      const uint32_t byc = (((gq < 4) ? vsc.x : vsc.y) >> bsh) & 0xffu;
      const uint32_t byd = (((gq < 4) ? vsd.x : vsd.y) >> bsh) & 0xffu;
      const uint32_t rv01 = pow2_neg_f16((int)eva - (int)bya) | (pow2_neg_f16((int)evb - (int)byb) << 16);
      const uint32_t rv89 = pow2_neg_f16((int)evc - (int)byc) | (pow2_neg_f16((int)evd - (int)byd) << 16);
      // V exponents of tokens gq and gq+8 come from lane c' = gq / 2
      const uint32_t evpack = eva | (evb << 8) | (evc << 16) | (evd << 24);
      const uint32_t evsrc = __shfl_sync(0xffffffffu, evpack, gq >> 1);
      const int ev0 = (int)((evsrc >> (8 * (gq & 1))) & 0xffu);
      const int ev1 = (int)((evsrc >> (16 + 8 * (gq & 1))) & 0xffu);

      // -- scores and online softmax
      const float fk0 = scale_log2e * ue8m0_to_f32(ek0);
      const float fk1 = scale_log2e * ue8m0_to_f32(ek1);
      const bool v0 = gq < nvalid, v1 = gq + 8 < nvalid;
      uint32_t pw[NT][2];
      bool rescale = false;
      float alpha_o[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float w4[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float s0 = v0 ? sacc[nt][h] * fk0 : -INFINITY;
          const float s1 = v1 ? sacc[nt][2 + h] * fk1 : -INFINITY;
          const float u0 = s0 + (float)(ev0 - 127);
          const float u1 = s1 + (float)(ev1 - 127);
          float tmax = fmaxf(s0, s1), umax = fmaxf(u0, u1);
#pragma unroll
          for (int msk = 4; msk < 32; msk <<= 1) {
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, msk));
            umax = fmaxf(umax, __shfl_xor_sync(0xffffffffu, umax, msk));
          }
          const float m_new = fmaxf(m_run[nt][h], tmax);
          const float mu_new = fmaxf(mu_run[nt][h], umax);
          l_run[nt][h] = l_run[nt][h] * fast_exp2(m_run[nt][h] - m_new) + fast_exp2(s0 - m_new) +
                         fast_exp2(s1 - m_new);
          alpha_o[nt][h] = fast_exp2(mu_run[nt][h] - mu_new);
          rescale |= mu_new != mu_run[nt][h];
          m_run[nt][h] = m_new;
          mu_run[nt][h] = mu_new;
          w4[h] = fast_exp2(u0 - mu_new);
          w4[2 + h] = fast_exp2(u1 - mu_new);
        }
        pw[nt][0] = movmatrix_trans(pack_f16x2(w4[0], w4[1]));
        pw[nt][1] = movmatrix_trans(pack_f16x2(w4[2], w4[3]));
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 16; ++mt) {
            o[nt][mt][0] *= alpha_o[nt][0];
            o[nt][mt][1] *= alpha_o[nt][1];
            o[nt][mt][2] *= alpha_o[nt][0];
            o[nt][mt][3] *= alpha_o[nt][1];
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
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t a0 = hmul2(A0[e], rv01), a1 = hmul2(A1[e], rv01);
          const uint32_t a2 = hmul2(A2[e], rv89), a3 = hmul2(A3[e], rv89);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16_16816(o[nt][4 * q + e], a0, a1, a2, a3, pw[nt][0], pw[nt][1]);
        }
      }
    }
    __syncwarp();
    if (j + NSTAGE < n_my) issue(j + NSTAGE);
  }
  if (timed_out) {
    if (lane == 0) atomicOr(err, kErrTimeout);
    // wait (bounded) for this warp's copies still in flight before leaving
    for (int jj = j; jj < n_my && jj < j + NSTAGE; ++jj)
      (void)mbar_wait(bar_base + 8 * (jj % NSTAGE), (uint32_t)((jj / NSTAGE) & 1));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        m_run[nt][h] = -INFINITY;
        mu_run[nt][h] = -INFINITY;
        l_run[nt][h] = 0.f;
      }
  }
  // full row sums over the 8 lanes that share c
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1)
        l_run[nt][h] += __shfl_xor_sync(0xffffffffu, l_run[nt][h], msk);

  // ---- merge the warps' states: partial (o, lse) of this split -------------
  __syncthreads();  // every warp is done with its stage buffers
  float* osm = reinterpret_cast<float*>(smem);
  float* stats = reinterpret_cast<float*>(smem + Lay::kStatsOff);
  float* rowinfo = reinterpret_cast<float*>(smem + Lay::kRowInfoOff);
  float* my_o = osm + warp * Lay::kRows * Lay::kORowStride;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r0 = nt * 8 + 2 * c;
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) {
      const int d = 32 * gq + 2 * mt;
      *reinterpret_cast<float2*>(my_o + r0 * Lay::kORowStride + d) = make_float2(o[nt][mt][0], o[nt][mt][2]);
      *reinterpret_cast<float2*>(my_o + (r0 + 1) * Lay::kORowStride + d) = make_float2(o[nt][mt][1], o[nt][mt][3]);
    }
    if (gq == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float* st = stats + (warp * Lay::kRows + r0 + h) * 4;
        st[0] = m_run[nt][h];
        st[1] = mu_run[nt][h];
        st[2] = l_run[nt][h];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < QG) {
    const int r = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, stats[(w * Lay::kRows + r) * 4]);
    float Ls = 0.f;
    for (int w = 0; w < NWARPS; ++w) {
      const float* st = stats + (w * Lay::kRows + r) * 4;
      if (st[2] > 0.f) Ls += st[2] * fast_exp2(st[0] - M);
    }
    float* ri = rowinfo + r * (NWARPS + 2);
    for (int w = 0; w < NWARPS; ++w) {
      const float* st = stats + (w * Lay::kRows + r) * 4;
      ri[w] = (Ls > 0.f && st[2] > 0.f) ? fast_exp2(st[1] - M) / Ls : 0.f;
    }
    ri[NWARPS] = Ls > 0.f ? M + fast_log2(Ls) : -INFINITY;
    part_lse[((int64_t)(b * Hq + g * QG + r)) * S + split] = ri[NWARPS];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < QG * (kHeadDim / 4); idx += NWARPS * 32) {
    const int r = idx / (kHeadDim / 4), d4 = (idx % (kHeadDim / 4)) * 4;
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
    *reinterpret_cast<float4*>(part_o + (((int64_t)(b * Hq + g * QG + r)) * S + split) * kHeadDim + d4) = acc;
  }
}

// Stage 2: merge the active splits of each (sequence, query head).
__global__ void __launch_bounds__(128)
decode_stage2(const float* __restrict__ part_o, const float* __restrict__ part_lse,
              const int32_t* __restrict__ seq_lens, int B, int Hq, int S, int max_blocks,
              uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= B * Hq) return;
  const int b = row / Hq;
  const int L = clamp_len(seq_lens[b], max_blocks);
  const SplitPlan plan = split_plan(L, S);
  const int n = plan.n_active;
  const float* lse = part_lse + (int64_t)row * S;
  float mx = -INFINITY;
  for (int s = lane; s < n; s += 32) mx = fmaxf(mx, lse[s]);
#pragma unroll
  for (int msk = 16; msk > 0; msk >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float den = 0.f;
  if (n > 0 && mx > -INFINITY) {
    const float* po = part_o + (int64_t)row * S * kHeadDim + lane * 8;
    for (int s0 = 0; s0 < n; s0 += 32) {
      const float wl = (s0 + lane < n) ? fast_exp2(lse[s0 + lane] - mx) : 0.f;
      const int cnt = min(32, n - s0);
      for (int k = 0; k < cnt; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, k);
        den += w;
        const float4 v0 = *reinterpret_cast<const float4*>(po + (int64_t)(s0 + k) * kHeadDim);
        const float4 v1 = *reinterpret_cast<const float4*>(po + (int64_t)(s0 + k) * kHeadDim + 4);
        acc[0] += w * v0.x; acc[1] += w * v0.y; acc[2] += w * v0.z; acc[3] += w * v0.w;
        acc[4] += w * v1.x; acc[5] += w * v1.y; acc[6] += w * v1.z; acc[7] += w * v1.w;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(acc[2 * i + 1] * inv), "f"(acc[2 * i] * inv));
    pk[i] = r;
  }
  *reinterpret_cast<uint4*>(out + (int64_t)row * kHeadDim + lane * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

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

template <int NT>
static cudaError_t launch_stage1_t(const uint16_t* query, int64_t q_ss, int64_t q_sh,
                                   const uint8_t* kv, const int32_t* bt, const int32_t* sl,
                                   float scale, int B, int Hq, int Hk, int num_blocks,
                                   int max_blocks, int S, float* part_o, float* part_lse,
                                   unsigned* err, cudaStream_t stream) {
  constexpr int NWARPS = 4, NSTAGE = 3;
  using Lay = Stage1Layout<NT, NWARPS, NSTAGE>;
  auto kern = decode_stage1<NT, NWARPS, NSTAGE>;
  static int configured_mask = 0;  // one bit per device (first 31 devices)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_mask |= 1 << dev;
  }
  dim3 grid(S, Hk, B);
  kern<<<grid, NWARPS * 32, Lay::kBytes, stream>>>(query, q_ss, q_sh, kv, bt, sl, scale * kLog2e,
                                                   Hq, Hk, Hq / Hk, num_blocks, max_blocks, S,
                                                   part_o, part_lse, err);
  return cudaGetLastError();
}

cudaError_t launch_decode(const uint16_t* query, int64_t q_ss, int64_t q_sh, const uint8_t* kv,
                          const int32_t* bt, const int32_t* sl, float scale, int B, int Hq,
                          int Hk, int num_blocks, int max_blocks, int S, void* workspace,
                          uint16_t* out, unsigned* err, cudaStream_t stream,
                          cudaEvent_t ev_before_stage1, cudaEvent_t ev_after_stage1) {
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = part_o + (size_t)B * Hq * S * kHeadDim;
  const int QG = Hq / Hk;
  if (ev_before_stage1) {
    cudaError_t er = record_timing_event(ev_before_stage1, stream);
    if (er != cudaSuccess) return er;
  }
  cudaError_t e = (QG == 16)
      ? launch_stage1_t<2>(query, q_ss, q_sh, kv, bt, sl, scale, B, Hq, Hk, num_blocks, max_blocks, S, part_o, part_lse, err, stream)
      : launch_stage1_t<1>(query, q_ss, q_sh, kv, bt, sl, scale, B, Hq, Hk, num_blocks, max_blocks, S, part_o, part_lse, err, stream);
  if (e != cudaSuccess) return e;
  if (ev_after_stage1) {
    e = record_timing_event(ev_after_stage1, stream);
    if (e != cudaSuccess) return e;
  }
  const int rows = B * Hq;
  decode_stage2<<<(rows + 3) / 4, 128, 0, stream>>>(part_o, part_lse, sl, B, Hq, S, max_blocks, out);
  return cudaGetLastError();
}

}  // namespace uq
