// uq_device.cuh -- device-side helpers shared by the store and decode kernels:
// documented PTX conversions (E2M1, E4M3, f16), warp MMA, bulk async copies
// and bounded mbarrier waits.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace uq {

constexpr int kHeadDim = 256;
constexpr int kSlotBytes = 272;          // 128 K codes + 128 V codes + 8 + 8 scales
constexpr int kKScaleOff = 256;
constexpr int kVScaleOff = 264;
constexpr int kVCodeOff = 128;

// Bounded waits: each try_wait may suspend the thread for up to
// kWaitSuspendNs (it returns as soon as the phase completes), and a wait
// gives up after kWaitSpinLimit tries (about two seconds), sets
// UQ_DEVERR_TIMEOUT and lets the kernel return instead of hanging.  A test
// build shortens both (UQ_WAIT_SUSPEND_NS, UQ_WAIT_SPIN_LIMIT).
#ifndef UQ_WAIT_SUSPEND_NS
#define UQ_WAIT_SUSPEND_NS (1u << 16)
#endif
#ifndef UQ_WAIT_SPIN_LIMIT
#define UQ_WAIT_SPIN_LIMIT (1u << 15)
#endif
constexpr uint32_t kWaitSuspendNs = UQ_WAIT_SUSPEND_NS;
constexpr uint32_t kWaitSpinLimit = UQ_WAIT_SPIN_LIMIT;

constexpr unsigned kErrBadPage = 1u;
constexpr unsigned kErrBadSlot = 2u;
constexpr unsigned kErrTimeout = 4u;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Eight fp32 -> one word of eight E2M1 codes, element i in nibble i (bits
// 4i..4i+3).  Round to nearest even, saturating at +-6 (cvt ... satfinite);
// the conversion keeps the sign bit of a negative value that rounds to zero.
__device__ __forceinline__ uint32_t e2m1x8_from_f32(const float (&y)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(r)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  return r;
}

// Four bytes of a word, each two E2M1 codes -> four f16x2 registers.
__device__ __forceinline__ void f16x2x4_from_e2m1_word(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// Two fp32 -> E4M3 (round to nearest even, saturating at +-448) -> f16x2
// holding those E4M3 values exactly; `lo` lands in the low half.
__device__ __forceinline__ uint32_t e4m3_roundtrip_f16x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// D = A * B + D, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float fast_log2(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// 2^(byte - 127) as fp32, exact for every byte in [0, 254] (byte 0 is the
// subnormal 2^-127).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(1u << 22);
}

// 2^(13 - d) as f16 for the two halfwords d0, d1 of d2 (each 0..255),
// packed as f16x2: the biased exponent 28 - d in bits 14..10 of each half.
// A token's largest block (d = 0) maps to 2^13, so an E2M1 code times the
// factor stays below 6 * 2^13 = 49152, inside f16's range.  d >= 28 gives +0:
// a block 2^28 or more below its token's largest block is left to the
// caller; every kept factor is a normal f16, so the product c * 2^(13 - d)
// of an E2M1 code c stays exact.
constexpr uint32_t kRelSpan = 28;    // kept block exponents: d = 0 .. kRelSpan - 1
constexpr int kRelTop = 13;          // the largest block maps to 2^kRelTop
__device__ __forceinline__ uint32_t pow2_rel_f16x2(uint32_t d2) {
  uint32_t m;
  asm("min.u16x2 %0, %1, %2;" : "=r"(m) : "r"(d2), "r"(kRelSpan * 0x00010001u));
  return (kRelSpan * 0x00010001u - m) << 10;   // 28 - m for m in 0..28, no borrow
}

// 2^(byte - 127 - kRelTop) as fp32 for a block byte (exact; normal for
// byte >= 14, subnormal below).
__device__ __forceinline__ float ue8m0_rel_to_f32(uint32_t byte) {
  return byte >= 14u ? __uint_as_float((byte - 13u) << 23) : __uint_as_float(1u << (byte + 9u));
}

// Largest of the eight bytes of (lo, hi): the bytes spread over 16-bit
// lanes (native lane-wise integer max), three lane-wise maxima, then the
// larger lane.
__device__ __forceinline__ uint32_t max_byte8(uint32_t lo, uint32_t hi) {
  uint32_t m;
  asm("{\n\t.reg .b32 a, b, c, d;\n\t"
      "prmt.b32 a, %1, 0, 0x4240;\n\tprmt.b32 b, %1, 0, 0x4341;\n\t"
      "prmt.b32 c, %2, 0, 0x4240;\n\tprmt.b32 d, %2, 0, 0x4341;\n\t"
      "max.u16x2 a, a, b;\n\tmax.u16x2 c, c, d;\n\tmax.u16x2 %0, a, c;\n}\n"
      : "=r"(m) : "r"(lo), "r"(hi));
  return max(m & 0xffffu, m >> 16);
}

// True if any of the eight halfwords of four f16x2 relative scales (from
// pow2_rel_f16x2) is +0, i.e. some block lies 2^kRelSpan or more below its
// token's largest block.
__device__ __forceinline__ bool any_rel_zero(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t p3) {
  uint32_t m;
  asm("{\n\t.reg .b32 t;\n\tmin.u16x2 t, %1, %2;\n\tmin.u16x2 %0, %3, %4;\n\tmin.u16x2 %0, %0, t;\n}\n"
      : "=r"(m) : "r"(p0), "r"(p1), "r"(p2), "r"(p3));
  return min(m & 0xffffu, m >> 16) == 0u;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and bulk async copies (TMA engine).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false if the iteration cap ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kWaitSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(bar), "r"(parity), "r"(kWaitSuspendNs) : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Tiled TMA load of a 3-D box (coordinates x innermost) into shared memory,
// completing on mbarrier `bar`.  The tensor map lives in kernel parameter
// space (__grid_constant__); all operands are warp-uniform.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tensor_map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 ldg_nc_128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream still
// runs; pdl_wait blocks until that kernel has finished and its writes are
// visible (a no-op for a kernel launched without the attribute), and
// pdl_launch_dependents lets the next such kernel start early.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Tensor memory (TMEM) as per-thread storage.  One warp of the CTA allocates
// the columns (all 128 lanes) and publishes the base address in shared memory;
// warp w may then read and write only lanes 32 (w % 4) .. 32 (w % 4) + 31.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of the thread's own lane (shape 32x32b, x32).
// The wait is in the same statement, so the registers are valid on return.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
               "tcgen05.wait::ld.sync.aligned;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]) : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The reverse; complete it with tmem_wait_st before reading the columns back.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])) : "memory");
}

// Split form for overlapping a load with other work: issue 16 columns, then
// tmem_ld16_wait on the same registers before reading them.  The wait takes
// the registers as in-out operands, so no use of them moves above it.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, float (&v)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15]) : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_ld16_wait(float (&v)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]) :: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace uq
