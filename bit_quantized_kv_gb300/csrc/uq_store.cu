// uq_store.cu -- the store kernels: rotate K by the 256-point Hadamard matrix
// and pack K and V of each (token, kv head) into one 272-byte FP4 slot
// (vllm.v1.attention.backends.ultraquant_attn, UltraQuantAttentionImpl:
// _store_kv packs "K+V into FP4/UE8M0 slots" after rotating K by PiT).
//
// Work unit: one (token, kv head) row per group of 8 lanes.  The fast
// Walsh-Hadamard butterfly runs its stages in the fixed order
// h = 1, 2, ..., 128; every stage maps a pair (a, b) with a at the lower
// index to (a + b, a - b), so the fp32 result is the canonical one bit for
// bit whichever stages run in registers and which across lanes.
//
// bf16 path (store_bf16_kernel): lane g of a group loads the 16-byte chunks
// 8i + g (i = 0..3) of the row, so each load instruction reads 128
// contiguous bytes per row and uses every sector it touches; lane g then
// holds elements 64i + 8g + e (e = 0..7) in x[8i + e].  Stages h = 1, 2, 4
// and 64, 128 run in registers, h = 8, 16, 32 across the 8 lanes with
// shuffles.  UE8M0 block j = d / 32 of element d = 64i + 8g + e is 2i + g / 4,
// so a block's 32 values sit in register group i of 4 lanes and its amax
// takes two shuffles.  Each lane writes the 8 codes of each register group
// as one 4-byte word (bytes 32i + 4g of the code array).
//
// fp32 pre-rotated path (store_rotated_f32_kernel): lane g owns elements [32g, 32g+32),
// exactly the g-th UE8M0 block, and writes 16 code bytes at once.
#include "uq_device.cuh"

namespace uq {

constexpr int kStoreThreads = 256;
constexpr int kLanesPerRow = 8;
constexpr int kRowsPerBlock = kStoreThreads / kLanesPerRow;

// Quantise 32 fp32 values (one UE8M0 block) into 16 code bytes + 1 scale byte.
__device__ __forceinline__ uint32_t quantize_block32(const float (&x)[32], uint4& codes) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  // shared exponent floor(log2 amax) - 2, clamped at -127: byte = max(biased - 2, 0)
  int biased = (int)(__float_as_uint(amax) >> 23);
  uint32_t byte = (uint32_t)max(biased - 2, 0);
  // 2^-(byte - 127) = 2^(127 - byte): biased exponent 254 - byte, always normal
  const float inv = __uint_as_float((254u - byte) << 23);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = x[q * 8 + e] * inv;
    w[q] = e2m1x8_from_f32(y);
  }
  codes = make_uint4(w[0], w[1], w[2], w[3]);
  return byte;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float* x) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_bits_to_f32(u[i] & 0xffffu);
    x[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
  }
}

// Canonical FWHT of the 256 values of a row in the bf16 path's layout
// (lane g: elements 64i + 8g + e in x[8i + e]).
__device__ __forceinline__ void fwht256_interleaved(float (&x)[32], int glane) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {          // element strides 1, 2, 4
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < kLanesPerRow; m <<= 1) {   // element strides 8, 16, 32
    const float sgn = (glane & m) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = fmaf(x[i], sgn, other);
    }
  }
#pragma unroll
  for (int h = 8; h < 32; h <<= 1) {         // element strides 64, 128
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
}

// Quantise one row half (K or V) held in the bf16 path's layout and, when
// do_row, write its 128 code bytes and 8 scale bytes at dst + code_off and
// dst + scale_off.  Every lane joins the shuffles.
__device__ __forceinline__ void quantize_interleaved(const float (&x)[32], int glane, uint8_t* dst,
                                                     int code_off, int scale_off, bool do_row) {
  uint32_t bytes[4], w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[8 * i + e]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));   // the block's 4 lanes
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // shared exponent floor(log2 amax) - 2, clamped at -127: byte = max(biased - 2, 0)
    const int biased = (int)(__float_as_uint(amax) >> 23);
    const uint32_t byte = (uint32_t)max(biased - 2, 0);
    const float inv = __uint_as_float((254u - byte) << 23);   // 2^(127 - byte), normal
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = x[8 * i + e] * inv;
    w[i] = e2m1x8_from_f32(y);
    bytes[i] = byte;
  }
  if (!do_row) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(dst + code_off + 32 * i + 4 * glane) = w[i];
  // lane g writes the scale of block 2 (g % 4) + g / 4, which it holds in group g % 4
  const int gi = glane & 3;
  const uint32_t b = gi == 0 ? bytes[0] : gi == 1 ? bytes[1] : gi == 2 ? bytes[2] : bytes[3];
  dst[scale_off + 2 * gi + (glane >> 2)] = (uint8_t)b;
}

__device__ __forceinline__ uint4 ldg_nc_l1_128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// key/value are bf16 [N] rows of [Hk][256] at the given token strides.
__global__ void __launch_bounds__(kStoreThreads)
store_bf16_kernel(const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
                  uint8_t* __restrict__ kv_cache, const int64_t* __restrict__ slot_mapping,
                  int64_t num_rows, int Hk, int64_t key_stride, int64_t value_stride,
                  int64_t num_slots, unsigned* __restrict__ err) {
  pdl_launch_dependents();   // a decode plan queued behind the store may be scheduled now
  const int lane = threadIdx.x & 31;
  const int glane = lane & (kLanesPerRow - 1);
  const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 3);
  const bool active = row < num_rows;
  const int64_t n = active ? row / Hk : 0;
  const int h = active ? (int)(row - n * Hk) : 0;
  const int64_t slot = active ? slot_mapping[n] : -1;
  const bool in_range = slot < num_slots;
  if (active && slot >= 0 && !in_range && glane == 0) atomicOr(err, kErrBadSlot);
  // Inactive groups still join the (full-warp) shuffles below.
  const bool do_row = active && slot >= 0 && in_range;

  const uint16_t* kp = key + n * key_stride + (int64_t)h * kHeadDim + 8 * glane;
  const uint16_t* vp = value + n * value_stride + (int64_t)h * kHeadDim + 8 * glane;
  float k[32], v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // L1-allocating: the group's 4 loads of a row share no sector, but the
    // warp's requests then leave L1 as whole lines.
    const uint4 kq = do_row ? ldg_nc_l1_128(kp + 64 * i) : make_uint4(0, 0, 0, 0);
    const uint4 vq = do_row ? ldg_nc_l1_128(vp + 64 * i) : make_uint4(0, 0, 0, 0);
    unpack_bf16x8(kq, k + 8 * i);
    unpack_bf16x8(vq, v + 8 * i);
  }
  fwht256_interleaved(k, glane);
#pragma unroll
  for (int i = 0; i < 32; ++i) k[i] = k[i] * 0.0625f;   // exact: power of two
  // slot = page * block_size + offset, so the cache row is slot * Hk + h
  uint8_t* dst = kv_cache + (slot * Hk + h) * (int64_t)kSlotBytes;
  quantize_interleaved(k, glane, dst, 0, kKScaleOff, do_row);
  quantize_interleaved(v, glane, dst, kVCodeOff, kVScaleOff, do_row);
}

// key/value are fp32 [N][Hk][256] with K already rotated.
__global__ void __launch_bounds__(kStoreThreads)
store_rotated_f32_kernel(const float* __restrict__ key, const float* __restrict__ value,
                         uint8_t* __restrict__ kv_cache, const int64_t* __restrict__ slot_mapping,
                         int64_t num_rows, int Hk, int64_t num_slots, unsigned* __restrict__ err) {
  pdl_launch_dependents();   // a decode plan queued behind the store may be scheduled now
  const int lane = threadIdx.x & 31;
  const int glane = lane & (kLanesPerRow - 1);
  const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 3);
  if (row >= num_rows) return;   // no shuffles below
  const int64_t n = row / Hk;
  const int h = (int)(row - n * Hk);
  const int64_t slot = slot_mapping[n];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (glane == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  float k[32], v[32];
  const float* kp = key + row * kHeadDim + glane * 32;
  const float* vp = value + row * kHeadDim + glane * 32;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 kq = ldg_nc_128(kp + 4 * q);
    const uint4 vq = ldg_nc_128(vp + 4 * q);
    k[4 * q] = __uint_as_float(kq.x); k[4 * q + 1] = __uint_as_float(kq.y);
    k[4 * q + 2] = __uint_as_float(kq.z); k[4 * q + 3] = __uint_as_float(kq.w);
    v[4 * q] = __uint_as_float(vq.x); v[4 * q + 1] = __uint_as_float(vq.y);
    v[4 * q + 2] = __uint_as_float(vq.z); v[4 * q + 3] = __uint_as_float(vq.w);
  }
  uint4 kc, vc;
  const uint32_t kbyte = quantize_block32(k, kc);
  const uint32_t vbyte = quantize_block32(v, vc);
  uint8_t* dst = kv_cache + (slot * Hk + h) * (int64_t)kSlotBytes;
  *reinterpret_cast<uint4*>(dst + 16 * glane) = kc;
  *reinterpret_cast<uint4*>(dst + kVCodeOff + 16 * glane) = vc;
  dst[kKScaleOff + glane] = (uint8_t)kbyte;
  dst[kVScaleOff + glane] = (uint8_t)vbyte;
}

cudaError_t launch_store(bool rotated_f32, const void* key, const void* value, void* kv_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int Hk,
                         int64_t key_stride, int64_t value_stride, int block_size,
                         int64_t num_slots, unsigned* err, cudaStream_t stream) {
  const int64_t rows = num_tokens * Hk;
  const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks <= 0) return cudaSuccess;
  if (rotated_f32)
    store_rotated_f32_kernel<<<(unsigned)blocks, kStoreThreads, 0, stream>>>(
        static_cast<const float*>(key), static_cast<const float*>(value),
        static_cast<uint8_t*>(kv_cache), slot_mapping, rows, Hk, num_slots, err);
  else
    store_bf16_kernel<<<(unsigned)blocks, kStoreThreads, 0, stream>>>(
        static_cast<const uint16_t*>(key), static_cast<const uint16_t*>(value),
        static_cast<uint8_t*>(kv_cache), slot_mapping, rows, Hk, key_stride, value_stride,
        num_slots, err);
  return cudaGetLastError();
}

}  // namespace uq
