// uq_dequant.cu -- full-prefix dequantisation of one sequence's pages to bf16
// (vllm.v1.attention.backends.ultraquant_attn,
// UltraQuantAttentionImpl._ultraquant_continuation_prefill: the prefix
// buffers (1, Hk, alloc_len, D) filled by ultraquant_full_dequant_kv before
// the dense prefill of a large continuation chunk).
//
// The kernel streams: 272 bytes read and 1024 bytes written per (token, kv
// head).  A CTA expands one (16-token tile, kv head); a page of block_size
// tokens is block_size / 16 tiles.  Each of the 8 warps takes two of the
// tile's 16 tokens, and for a token lane l converts elements
// 8l .. 8l+7 of K and of V: it reads one 32-bit word of codes from each code
// region (the warp reads each 128-byte region whole) and the scale byte of
// block l/4, and writes 16 bytes of each output row (the warp writes each
// 512-byte bf16 row whole).  Consecutive CTAs take neighbouring kv heads of
// the same page, whose slots are adjacent in the cache.
//
// Each value E2M1(c) * 2^(byte - 127) is formed exactly in fp32: the f16
// from the E2M1 conversion is exact, and the power of two is applied as two
// factors 2^floor(e/2) * 2^(e - floor(e/2)) that are both normal fp32
// numbers for every byte, so the one rounding happens at the end (only an
// overflow rounds: to inf).  The bf16 conversion is then exact.
#include <cuda_fp16.h>

#include "uq_device.cuh"

namespace uq {

constexpr int kDqPage = 16;
constexpr int kDqWarps = 8;                        // two tokens of the tile per warp

// 2^(byte - 127) as two normal fp32 factors.
__device__ __forceinline__ void scale_factors(uint32_t byte, float& f1, float& f2) {
  const int e = (int)byte - 127;
  const int e1 = e >> 1;             // floor(e / 2), in [-64, 64]
  const int e2 = e - e1;             // in [-63, 64]
  f1 = __uint_as_float((uint32_t)(127 + e1) << 23);
  f2 = __uint_as_float((uint32_t)(127 + e2) << 23);
}

// One word of 8 codes (element i in nibble i) and its scale byte -> 8 bf16.
__device__ __forceinline__ uint4 dequant_word8(uint32_t codes, uint32_t byte) {
  float f1, f2;
  scale_factors(byte, f1, f2);
  uint32_t h[4], r[4];
  f16x2x4_from_e2m1_word(codes, h);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
    const float lo = __fmul_rn(__fmul_rn(v.x, f1), f2);
    const float hi = __fmul_rn(__fmul_rn(v.y, f1), f2);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r[j]) : "f"(hi), "f"(lo));
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

__device__ __forceinline__ uint32_t ldg_nc_32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kDqWarps * 32)
full_dequant_kernel(const uint8_t* __restrict__ kv, const int32_t* __restrict__ block_table,
                    int n_tiles, int lg_tpp, int Hk, int num_blocks, uint16_t* __restrict__ k_out,
                    uint16_t* __restrict__ v_out, unsigned* __restrict__ err) {
  const int64_t item = blockIdx.x;                  // < n_tiles * Hk
  const int p = (int)(item / Hk), h = (int)(item - (int64_t)p * Hk);   // tile p of the sequence
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pid = block_table[p >> lg_tpp];
  const int64_t alloc_len = (int64_t)n_tiles * kDqPage;
  const int64_t row0 = (int64_t)h * alloc_len + (int64_t)p * kDqPage + 2 * warp;
  uint4* ko = reinterpret_cast<uint4*>(k_out + row0 * kHeadDim) + lane;
  uint4* vo = reinterpret_cast<uint4*>(v_out + row0 * kHeadDim) + lane;
  constexpr int kRowVec = kHeadDim / 8;             // uint4 per output row
  if ((unsigned)pid >= (unsigned)num_blocks) {
    if (threadIdx.x == 0) atomicOr(err, kErrBadPage);   // once per tile of the page
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    ko[0] = z;
    ko[kRowVec] = z;
    vo[0] = z;
    vo[kRowVec] = z;
    return;
  }
  const int64_t slot0 = ((int64_t)pid << (4 + lg_tpp)) + ((p & ((1 << lg_tpp) - 1)) << 4) + 2 * warp;
  const uint8_t* s0 = kv + (slot0 * Hk + h) * kSlotBytes;
  const uint8_t* s1 = s0 + (int64_t)Hk * kSlotBytes;   // the next token of the page
  const uint32_t k0 = ldg_nc_32(s0 + 4 * lane), v0 = ldg_nc_32(s0 + kVCodeOff + 4 * lane);
  const uint32_t k1 = ldg_nc_32(s1 + 4 * lane), v1 = ldg_nc_32(s1 + kVCodeOff + 4 * lane);
  const uint32_t kb0 = ldg_nc_u8(s0 + kKScaleOff + (lane >> 2)), vb0 = ldg_nc_u8(s0 + kVScaleOff + (lane >> 2));
  const uint32_t kb1 = ldg_nc_u8(s1 + kKScaleOff + (lane >> 2)), vb1 = ldg_nc_u8(s1 + kVScaleOff + (lane >> 2));
  ko[0] = dequant_word8(k0, kb0);
  vo[0] = dequant_word8(v0, vb0);
  ko[kRowVec] = dequant_word8(k1, kb1);
  vo[kRowVec] = dequant_word8(v1, vb1);
}

cudaError_t launch_full_dequant(const uint8_t* kv, const int32_t* block_table, int n_pages,
                                int lg_tpp, int Hk, int num_blocks, uint16_t* k_out, uint16_t* v_out,
                                unsigned* err, cudaStream_t stream) {
  const int n_tiles = n_pages << lg_tpp;
  const int64_t items = (int64_t)n_tiles * Hk;
  if (items <= 0) return cudaSuccess;
  full_dequant_kernel<<<(unsigned)items, kDqWarps * 32, 0, stream>>>(kv, block_table, n_tiles, lg_tpp,
                                                                    Hk, num_blocks, k_out, v_out, err);
  return cudaGetLastError();
}

}  // namespace uq
