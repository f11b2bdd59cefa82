// uq_store.cu -- the store kernel: rotate K by the 256-point Hadamard matrix
// and pack K and V of each (token, kv head) into one 272-byte FP4 slot
// (vllm.v1.attention.backends.ultraquant_attn, UltraQuantAttentionImpl:
// _store_kv packs "K+V into FP4/UE8M0 slots" after rotating K by PiT).
//
// Work unit: one (token, kv head) row per group of 8 lanes; lane j of the
// group owns elements [32j, 32j+32), which is exactly the j-th UE8M0 block.
// The fast Walsh-Hadamard butterfly runs its stages h = 1..16 inside each
// lane's registers and h = 32, 64, 128 across the 8 lanes with shuffles, in
// the fixed order h = 1, 2, ..., 128; every stage maps a pair (a, b) with a
// at the lower index to (a + b, a - b), so the fp32 result is the canonical
// one bit for bit.  The block amax is then lane-local.  Each lane writes its
// 32 codes of K and of V as one 16-byte store each, plus one scale byte each.
#include "uq_device.cuh"

namespace uq {

constexpr int kStoreThreads = 256;
constexpr int kLanesPerRow = 8;
constexpr int kRowsPerBlock = kStoreThreads / kLanesPerRow;

// Canonical FWHT of the 256 values held by the 8 lanes of a group
// (lane j: elements 32j .. 32j+31 in x[0..31]).
__device__ __forceinline__ void fwht256_group8(float (&x)[32], int glane) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
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
  for (int m = 1; m < kLanesPerRow; m <<= 1) {
    // lower lane holds a (own), upper lane holds b (own): (a + b, a - b).
    // fma(own, -1, other) rounds other - own exactly like a subtraction.
    const float sgn = (glane & m) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = fmaf(x[i], sgn, other);
    }
  }
}

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

// ROTATED_F32 = false: key/value are bf16 and K is rotated here.
// ROTATED_F32 = true : key/value are fp32 [N][Hk][256] and K is already rotated.
template <bool ROTATED_F32>
__global__ void __launch_bounds__(kStoreThreads)
store_kernel(const void* __restrict__ key, const void* __restrict__ value,
             uint8_t* __restrict__ kv_cache, const int64_t* __restrict__ slot_mapping,
             int64_t num_rows, int Hk, int64_t key_stride, int64_t value_stride,
             int block_size, int64_t num_slots, unsigned* __restrict__ err) {
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

  float k[32], v[32];
  if (!ROTATED_F32) {
    const uint16_t* kp = static_cast<const uint16_t*>(key) + n * key_stride + (int64_t)h * kHeadDim + glane * 32;
    const uint16_t* vp = static_cast<const uint16_t*>(value) + n * value_stride + (int64_t)h * kHeadDim + glane * 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 kq = do_row ? ldg_nc_128(kp + 8 * q) : make_uint4(0, 0, 0, 0);
      uint4 vq = do_row ? ldg_nc_128(vp + 8 * q) : make_uint4(0, 0, 0, 0);
      unpack_bf16x8(kq, k + 8 * q);
      unpack_bf16x8(vq, v + 8 * q);
    }
    fwht256_group8(k, glane);
#pragma unroll
    for (int i = 0; i < 32; ++i) k[i] = k[i] * 0.0625f;  // exact: power of two
  } else {
    const float* kp = static_cast<const float*>(key) + (n * Hk + h) * kHeadDim + glane * 32;
    const float* vp = static_cast<const float*>(value) + (n * Hk + h) * kHeadDim + glane * 32;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4 kq = do_row ? ldg_nc_128(kp + 4 * q) : make_uint4(0, 0, 0, 0);
      uint4 vq = do_row ? ldg_nc_128(vp + 4 * q) : make_uint4(0, 0, 0, 0);
      k[4 * q] = __uint_as_float(kq.x); k[4 * q + 1] = __uint_as_float(kq.y);
      k[4 * q + 2] = __uint_as_float(kq.z); k[4 * q + 3] = __uint_as_float(kq.w);
      v[4 * q] = __uint_as_float(vq.x); v[4 * q + 1] = __uint_as_float(vq.y);
      v[4 * q + 2] = __uint_as_float(vq.z); v[4 * q + 3] = __uint_as_float(vq.w);
    }
  }
  if (!do_row) return;

  uint4 kc, vc;
  const uint32_t kbyte = quantize_block32(k, kc);
  const uint32_t vbyte = quantize_block32(v, vc);
  const int64_t page = slot / block_size, off = slot - page * block_size;
  uint8_t* dst = kv_cache + ((page * block_size + off) * Hk + h) * (int64_t)kSlotBytes;
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
    store_kernel<true><<<(unsigned)blocks, kStoreThreads, 0, stream>>>(
        key, value, static_cast<uint8_t*>(kv_cache), slot_mapping, rows, Hk, key_stride,
        value_stride, block_size, num_slots, err);
  else
    store_kernel<false><<<(unsigned)blocks, kStoreThreads, 0, stream>>>(
        key, value, static_cast<uint8_t*>(kv_cache), slot_mapping, rows, Hk, key_stride,
        value_stride, block_size, num_slots, err);
  return cudaGetLastError();
}

}  // namespace uq
