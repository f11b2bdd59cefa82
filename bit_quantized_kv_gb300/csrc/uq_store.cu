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
// bf16 path (store_bf16_kernel): lane g of a group copies the 16-byte chunks
// 8i + g (i = 0..3) of the row's K and of its V, so each copy instruction
// reads 128 contiguous bytes per row and uses every sector it touches; lane
// g then holds elements 64i + 8g + e (e = 0..7) in x[8i + e].  Stages h = 1,
// 2, 4 and 64, 128 run in registers, h = 8, 16, 32 across the 8 lanes with
// shuffles; registers r and r + 16 travel as one packed fp32 pair, so all
// stages but h = 128 run two values per instruction.  UE8M0 block j = d / 32
// of element d = 64i + 8g + e is 2i + g / 4, so a block's 32 values sit in
// register group i of 4 lanes and its amax takes two shuffles.  Each lane
// writes the 8 codes of each register group as one 4-byte word (bytes
// 32i + 4g of the code array).
//
// The bf16 kernel is persistent (as many CTAs as fit on the GPU at once)
// and double-buffers its inputs in shared memory: each thread starts the
// asynchronous copies (cp.async) of its chunks of the next row before it
// rotates and quantises the current one, so the SM keeps reads in flight
// through the arithmetic.  The one-shot version of this kernel (load, then
// compute, one row per group) reached 80% of the measured HBM bandwidth;
// the staged one 85%, and with the packed butterfly 91%.
//
// fp32 pre-rotated path (store_rotated_f32_kernel): lane g owns elements [32g, 32g+32),
// exactly the g-th UE8M0 block, and writes 16 code bytes at once.
#include <mutex>

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
// (lane g: elements 64i + 8g + e in x[8i + e]), scaled by 1/16 (exact).
// Registers r and r + 16 travel as one packed pair, so every stage but the
// one between them (element stride 128) runs on pairs.
__device__ __forceinline__ void fwht256_interleaved_scaled(float (&x)[32], int glane) {
  float2 p[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) p[j] = make_float2(x[j], x[j + 16]);
  const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {          // element strides 1, 2, 4
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if ((j & h) == 0) {
        const float2 a = p[j], b = p[j + h];
        p[j] = __fadd2_rn(a, b);
        p[j + h] = __ffma2_rn(b, neg1, a);   // a - b
      }
    }
  }
#pragma unroll
  for (int m = 1; m < kLanesPerRow; m <<= 1) {   // element strides 8, 16, 32
    const float sg = (glane & m) ? -1.f : 1.f;
    const float2 sgn = make_float2(sg, sg);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, p[j].x, m),
                                       __shfl_xor_sync(0xffffffffu, p[j].y, m));
      p[j] = __ffma2_rn(p[j], sgn, other);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {              // element stride 64
    const float2 a = p[j], b = p[j + 8];
    p[j] = __fadd2_rn(a, b);
    p[j + 8] = __ffma2_rn(b, neg1, a);
  }
  const float2 sixteenth = make_float2(0.0625f, 0.0625f);
#pragma unroll
  for (int j = 0; j < 16; ++j) {             // element stride 128, then the 1/16
    const float a = p[j].x, b = p[j].y;
    p[j] = __fmul2_rn(make_float2(a + b, a - b), sixteenth);
    x[j] = p[j].x;
    x[j + 16] = p[j].y;
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
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 t = __fmul2_rn(make_float2(x[8 * i + e], x[8 * i + e + 1]), inv2);
      y[e] = t.x;
      y[e + 1] = t.y;
    }
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

// Resident CTAs per SM the bf16 kernel is built for: 80 registers per
// thread and 64 KB of staging per CTA both allow three.
constexpr int kStoreMinBlocks = 3;
// Shared staging of one row's inputs per thread: 8 chunks of 16 B (K 0..3,
// V 4..7), chunk-major so that a warp's 16-byte accesses are contiguous;
// two stages (the row being worked on and the next).
constexpr int kChunkStride = kStoreThreads * 16;
constexpr int kStoreStageBytes = 8 * kChunkStride;
constexpr int kStoreSmemBytes = 2 * kStoreStageBytes;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;   // a zero source size fills 16 zero bytes and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// key/value are bf16 [N] rows of [Hk][256] at the given token strides.
// Persistent: a warp takes rows w0 + (lane / 8), w0 + stride + (lane / 8), ...
// and each thread copies its chunks of the next row into shared memory
// (cp.async) before it works on the current one, so that an SM keeps reads
// in flight while its warps rotate and quantise.
__global__ void __launch_bounds__(kStoreThreads, kStoreMinBlocks)
store_bf16_kernel(const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
                  uint8_t* __restrict__ kv_cache, const int64_t* __restrict__ slot_mapping,
                  int64_t num_rows, int Hk, int64_t key_stride, int64_t value_stride,
                  int64_t num_slots, unsigned* __restrict__ err) {
  extern __shared__ __align__(16) uint8_t smem[];
  pdl_launch_dependents();   // a decode plan queued behind the store may be scheduled now
  const int lane = threadIdx.x & 31;
  const int glane = lane & (kLanesPerRow - 1);
  const int64_t stride = (int64_t)gridDim.x * kRowsPerBlock;
  // the warp's first row (uniform over the warp) and this group's row
  int64_t w0 = (int64_t)blockIdx.x * kRowsPerBlock + ((threadIdx.x >> 5) << 2);
  int64_t row = w0 + (lane >> 3);
  int64_t n = row / Hk;
  int h = (int)(row - n * Hk);
  const int64_t dn = stride / Hk;
  const int dh = (int)(stride - dn * Hk);
  // chunk c of stage s of this thread at my + s * kStoreStageBytes + c * kChunkStride
  const uint32_t my = smem_u32(smem) + threadIdx.x * 16;

  int64_t slot = -1;
  int stage = 0;
  // Rows past the end copy nothing (zero fill); a row with a negative slot
  // still copies its K and V (valid input rows), so no copy waits on the slot.
  auto fetch = [&](int s) {
    const bool act = row < num_rows;
    slot = act ? slot_mapping[n] : -1;
    const uint16_t* kp = key + (act ? n * key_stride + (int64_t)h * kHeadDim + 8 * glane : 0);
    const uint16_t* vp = value + (act ? n * value_stride + (int64_t)h * kHeadDim + 8 * glane : 0);
    const uint32_t base = my + s * kStoreStageBytes;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cp_async16(base + i * kChunkStride, kp + 64 * i, act);
      cp_async16(base + (4 + i) * kChunkStride, vp + 64 * i, act);
    }
    cp_async_commit();
  };
  fetch(0);
  for (; w0 < num_rows; w0 += stride) {
    cp_async_wait_all();   // this thread's chunks of the current row are in
    const uint32_t cur = my + stage * kStoreStageBytes;
    float k[32], v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack_bf16x8(lds128(cur + i * kChunkStride), k + 8 * i);
    const bool active = row < num_rows;
    const int64_t cur_slot = slot;
    const int cur_h = h;
    const bool in_range = cur_slot < num_slots;
    if (active && cur_slot >= 0 && !in_range && glane == 0) atomicOr(err, kErrBadSlot);
    // Inactive groups still join the (full-warp) shuffles below.
    const bool do_row = active && cur_slot >= 0 && in_range;
    // the next row of this group, copied into the other stage
    row += stride;
    n += dn;
    h += dh;
    if (h >= Hk) {
      h -= Hk;
      ++n;
    }
    fetch(stage ^ 1);

    fwht256_interleaved_scaled(k, glane);
    // slot = page * block_size + offset, so the cache row is slot * Hk + h
    uint8_t* dst = kv_cache + (cur_slot * Hk + cur_h) * (int64_t)kSlotBytes;
    quantize_interleaved(k, glane, dst, 0, kKScaleOff, do_row);
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack_bf16x8(lds128(cur + (4 + i) * kChunkStride), v + 8 * i);
    quantize_interleaved(v, glane, dst, kVCodeOff, kVScaleOff, do_row);
    stage ^= 1;
  }
  cp_async_wait_all();   // the last (empty) group
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

cudaError_t current_context_id(unsigned long long* id);

// Resident CTAs of the bf16 store kernel on the current device (SMs times
// CTAs per SM), looked up once per device and context.
static std::mutex g_store_grid_mutex;
static cudaError_t store_grid(int* grid) {
  static int grid_of_device[64] = {0};
  static unsigned long long ctx_of_device[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  unsigned long long ctx = 0;
  if ((e = current_context_id(&ctx)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_store_grid_mutex);
  if (dev >= 0 && dev < 64 && grid_of_device[dev] > 0 && ctx_of_device[dev] == ctx) {
    *grid = grid_of_device[dev];
    return cudaSuccess;
  }
  int sms = 0, per_sm = 0;
  if ((e = cudaFuncSetAttribute(store_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStoreSmemBytes)) !=
      cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, store_bf16_kernel, kStoreThreads, kStoreSmemBytes)) !=
      cudaSuccess)
    return e;
  *grid = sms * (per_sm > 0 ? per_sm : 1);
  if (dev >= 0 && dev < 64) {
    grid_of_device[dev] = *grid;
    ctx_of_device[dev] = ctx;
  }
  return cudaSuccess;
}

cudaError_t launch_store(bool rotated_f32, const void* key, const void* value, void* kv_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int Hk,
                         int64_t key_stride, int64_t value_stride, int block_size,
                         int64_t num_slots, unsigned* err, cudaStream_t stream) {
  const int64_t rows = num_tokens * Hk;
  int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks <= 0) return cudaSuccess;
  if (!rotated_f32) {
    int resident = 0;
    const cudaError_t e = store_grid(&resident);
    if (e != cudaSuccess) return e;
    if (blocks > resident) blocks = resident;
  }
  if (rotated_f32)
    store_rotated_f32_kernel<<<(unsigned)blocks, kStoreThreads, 0, stream>>>(
        static_cast<const float*>(key), static_cast<const float*>(value),
        static_cast<uint8_t*>(kv_cache), slot_mapping, rows, Hk, num_slots, err);
  else
    store_bf16_kernel<<<(unsigned)blocks, kStoreThreads, kStoreSmemBytes, stream>>>(
        static_cast<const uint16_t*>(key), static_cast<const uint16_t*>(value),
        static_cast<uint8_t*>(kv_cache), slot_mapping, rows, Hk, key_stride, value_stride,
        num_slots, err);
  return cudaGetLastError();
}

}  // namespace uq
