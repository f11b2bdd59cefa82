// uq_api.cu -- host side of the C ABI declared in include/uq.h: argument
// validation, error reporting, the device error word, and kernel launches.
// Nothing here allocates device memory or synchronises, except
// uq_check_device_error, which is documented to.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "uq.h"
#include "uq_decode_common.cuh"

namespace uq {
cudaError_t launch_store(bool rotated_f32, const void* key, const void* value, void* kv_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int Hk,
                         int64_t key_stride, int64_t value_stride, int block_size,
                         int64_t num_slots, unsigned* err, cudaStream_t stream);
cudaError_t launch_decode(const uint16_t* query, int64_t q_ss, int64_t q_sh, const uint8_t* kv,
                          const int32_t* bt, const SeqRows& sl, float scale, const float* sinks,
                          int B, int Hq, int Hk, int num_blocks, int max_blocks, int S,
                          void* workspace, uint16_t* out, unsigned* err, cudaStream_t stream,
                          cudaEvent_t ev_before_stage1, cudaEvent_t ev_after_stage1);
size_t decode_workspace_bytes(int B, int Hq, int S);
cudaError_t current_context_id(unsigned long long* id);
cudaError_t launch_full_dequant(const uint8_t* kv, const int32_t* block_table, int n_pages,
                                int lg_tpp, int Hk, int num_blocks, uint16_t* k_out, uint16_t* v_out,
                                unsigned* err, cudaStream_t stream);
}  // namespace uq

namespace uq {
// Unique id (cuCtxGetId) of the calling thread's current CUDA context.  A
// thread with no current context yet gets the current device's primary
// context (cudaSetDevice initialises and binds it).  Caches keyed by this id
// are looked up again after a device reset.
cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  static cudaError_t init_error = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    init_error = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q);
    if (init_error == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) init_error = cudaErrorNotSupported;
    if (init_error != cudaSuccess) return;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    init_error = cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q);
    if (init_error == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) init_error = cudaErrorNotSupported;
    if (init_error == cudaSuccess) get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (init_error != cudaSuccess) return init_error;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}
}  // namespace uq

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;

thread_local char g_last_error[512] = "";
thread_local cudaEvent_t g_ev_before_stage1 = nullptr;
thread_local cudaEvent_t g_ev_after_stage1 = nullptr;

// The device error word.  Kernels receive its device address; host code
// obtains that address with cudaGetSymbolAddress, once per device and CUDA
// context (a device reset creates a new context, in which the module and its
// variables live at new addresses).
__device__ unsigned int g_device_error_word;
unsigned int* g_err_ptr[kMaxDevices] = {nullptr};
unsigned long long g_err_ctx[kMaxDevices] = {0};
std::mutex g_err_mutex;

uq_status fail(uq_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

uq_status ok() {
  g_last_error[0] = '\0';
  return UQ_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Page sizes the decode and dequant kernels walk in whole 16-token tiles.
bool block_size_ok(int bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256; }

int log2_tiles_per_page(int bs) {
  int lg = 0;
  while ((16 << lg) < bs) ++lg;
  return lg;
}

// Device address of the error word in the current context (looked up on the
// first use in each context).
uq_status error_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(UQ_ERR_UNSUPPORTED, "device index %d >= %d", dev, kMaxDevices);
  unsigned long long ctx = 0;
  if ((e = uq::current_context_id(&ctx)) != cudaSuccess)
    return fail(UQ_ERR_CUDA, "reading the current context: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (!g_err_ptr[dev] || g_err_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error_word);
    if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
    g_err_ctx[dev] = ctx;
  }
  *out = g_err_ptr[dev];
  return UQ_OK;
}

uq_status check_store_args(const void* key, const void* value, void* kv_cache,
                           const int64_t* slot_mapping, int64_t num_tokens, int Hk, int D,
                           int num_blocks, int block_size, int slot_bytes, size_t elem_bytes) {
  if (num_tokens < 0) return fail(UQ_ERR_INVALID_ARG, "num_tokens %lld < 0", (long long)num_tokens);
  if (D != uq::kHeadDim) return fail(UQ_ERR_UNSUPPORTED, "head_dim %d unsupported (only 256)", D);
  if (slot_bytes != uq::kSlotBytes) return fail(UQ_ERR_INVALID_ARG, "slot_bytes %d != 272", slot_bytes);
  if (Hk < 1) return fail(UQ_ERR_INVALID_ARG, "num_kv_heads %d < 1", Hk);
  if (num_blocks < 1 || block_size < 1)
    return fail(UQ_ERR_INVALID_ARG, "num_blocks %d / block_size %d must be >= 1", num_blocks, block_size);
  if (num_tokens == 0) return UQ_OK;
  if (!key || !value || !kv_cache || !slot_mapping)
    return fail(UQ_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16))
    return fail(UQ_ERR_INVALID_ARG, "key, value and kv_cache must be 16-byte aligned");
  if (!aligned(slot_mapping, 8)) return fail(UQ_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  if (num_tokens > (int64_t)1 << 40 || (int64_t)Hk * num_tokens > ((int64_t)1 << 36))
    return fail(UQ_ERR_INVALID_ARG, "num_tokens * num_kv_heads too large");
  (void)elem_bytes;
  return UQ_OK;
}

}  // namespace

namespace uq {
// Records an error message for uq_last_error() from another translation unit.
uq_status set_error(uq_status code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace uq

extern "C" {

int uq_version(void) { return kVersion; }

size_t uq_slot_bytes(int head_dim) {
  return head_dim == uq::kHeadDim ? (size_t)uq::kSlotBytes : 0;
}

size_t uq_decode_workspace_bytes(int B, int Hq, int head_dim, int max_num_kv_splits) {
  if (B < 1 || Hq < 1 || head_dim != uq::kHeadDim || max_num_kv_splits < 1 || max_num_kv_splits > 256)
    return 0;
  return uq::decode_workspace_bytes(B, Hq, max_num_kv_splits);
}

const char* uq_last_error(void) { return g_last_error; }

uq_status uq_set_timing_events(void* before_stage1, void* after_stage1) {
  g_ev_before_stage1 = static_cast<cudaEvent_t>(before_stage1);
  g_ev_after_stage1 = static_cast<cudaEvent_t>(after_stage1);
  return UQ_OK;
}

uq_status uq_store(const void* key, const void* value, void* kv_cache, const int64_t* slot_mapping,
                   int64_t num_tokens, int num_kv_heads, int head_dim, int num_blocks,
                   int block_size, int slot_bytes, int64_t key_stride_tok,
                   int64_t value_stride_tok, void* stream) {
  uq_status st = check_store_args(key, value, kv_cache, slot_mapping, num_tokens, num_kv_heads,
                                  head_dim, num_blocks, block_size, slot_bytes, 2);
  if (st != UQ_OK) return st;
  if (num_tokens == 0) return ok();
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (key_stride_tok < row || value_stride_tok < row || key_stride_tok % 8 || value_stride_tok % 8)
    return fail(UQ_ERR_INVALID_ARG, "token strides (%lld, %lld) must be >= Hk*D and multiples of 8",
                (long long)key_stride_tok, (long long)value_stride_tok);
  unsigned int* err = nullptr;
  if ((st = error_word(&err)) != UQ_OK) return st;
  cudaError_t e = uq::launch_store(false, key, value, kv_cache, slot_mapping, num_tokens,
                                   num_kv_heads, key_stride_tok, value_stride_tok, block_size,
                                   (int64_t)num_blocks * block_size, err,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "store launch: %s", cudaGetErrorString(e));
  return ok();
}

uq_status uq_store_rotated_f32(const float* key_rot, const float* value, void* kv_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                               int head_dim, int num_blocks, int block_size, int slot_bytes,
                               void* stream) {
  uq_status st = check_store_args(key_rot, value, kv_cache, slot_mapping, num_tokens, num_kv_heads,
                                  head_dim, num_blocks, block_size, slot_bytes, 4);
  if (st != UQ_OK) return st;
  if (num_tokens == 0) return ok();
  unsigned int* err = nullptr;
  if ((st = error_word(&err)) != UQ_OK) return st;
  cudaError_t e = uq::launch_store(true, key_rot, value, kv_cache, slot_mapping, num_tokens,
                                   num_kv_heads, 0, 0, block_size, (int64_t)num_blocks * block_size,
                                   err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "store launch: %s", cudaGetErrorString(e));
  return ok();
}

uq_status uq_full_dequant(const void* kv_cache, const int32_t* block_table, int n_pages,
                          void* k_out, void* v_out, int Hk, int head_dim, int num_blocks,
                          int block_size, int slot_bytes, void* stream) {
  if (head_dim != uq::kHeadDim) return fail(UQ_ERR_UNSUPPORTED, "head_dim %d unsupported (only 256)", head_dim);
  if (!block_size_ok(block_size))
    return fail(UQ_ERR_UNSUPPORTED, "block_size %d unsupported (16, 32, 64, 128 or 256)", block_size);
  if (slot_bytes != uq::kSlotBytes) return fail(UQ_ERR_INVALID_ARG, "slot_bytes %d != 272", slot_bytes);
  if (Hk < 1 || Hk > 256) return fail(UQ_ERR_UNSUPPORTED, "Hk %d outside [1, 256]", Hk);
  if (num_blocks < 1) return fail(UQ_ERR_INVALID_ARG, "num_blocks %d < 1", num_blocks);
  if (n_pages < 0 || (int64_t)n_pages * block_size >= ((int64_t)1 << 31) ||
      (int64_t)n_pages * (block_size / 16) * Hk >= ((int64_t)1 << 31))
    return fail(UQ_ERR_INVALID_ARG,
                "n_pages %d: need n_pages * block_size and n_pages * (block_size / 16) * Hk < 2^31", n_pages);
  if (n_pages == 0) return ok();
  if (!kv_cache || !block_table || !k_out || !v_out)
    return fail(UQ_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(kv_cache, 16) || !aligned(k_out, 16) || !aligned(v_out, 16) || !aligned(block_table, 4))
    return fail(UQ_ERR_INVALID_ARG, "kv_cache, k_out, v_out must be 16-byte aligned, block_table 4-byte");
  unsigned int* err = nullptr;
  uq_status st = error_word(&err);
  if (st != UQ_OK) return st;
  if ((int64_t)num_blocks * block_size >= ((int64_t)1 << 31))
    return fail(UQ_ERR_INVALID_ARG, "num_blocks * block_size must be < 2^31");
  cudaError_t e = uq::launch_full_dequant(static_cast<const uint8_t*>(kv_cache), block_table, n_pages,
                                          log2_tiles_per_page(block_size), Hk, num_blocks,
                                          static_cast<uint16_t*>(k_out),
                                          static_cast<uint16_t*>(v_out), err,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "full dequant launch: %s", cudaGetErrorString(e));
  return ok();
}

namespace {

// Checks shared by uq_decode and uq_decode_multi_query, in the order the
// error messages report them.  *noop is set for an empty batch, which returns
// UQ_OK before any pointer is looked at.
uq_status check_decode(const void* query, const void* kv_cache, const int32_t* block_table,
                       float scale, int max_num_kv_splits, const void* workspace,
                       size_t workspace_bytes, const void* out, int B, int Hq, int Hk,
                       int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
                       int slot_bytes, int64_t q_stride_seq, int64_t q_stride_head, bool* noop) {
  *noop = false;
  if (B < 0) return fail(UQ_ERR_INVALID_ARG, "B %d < 0", B);
  if (head_dim != uq::kHeadDim) return fail(UQ_ERR_UNSUPPORTED, "head_dim %d unsupported (only 256)", head_dim);
  if (slot_bytes != uq::kSlotBytes) return fail(UQ_ERR_INVALID_ARG, "slot_bytes %d != 272", slot_bytes);
  if (!block_size_ok(block_size))
    return fail(UQ_ERR_UNSUPPORTED, "block_size %d unsupported (16, 32, 64, 128 or 256)", block_size);
  if (Hk < 1 || Hq < 1 || Hq % Hk) return fail(UQ_ERR_INVALID_ARG, "Hq %d must be a positive multiple of Hk %d", Hq, Hk);
  const int QG = Hq / Hk;
  if (QG != 6 && QG != 8 && QG != 16) return fail(UQ_ERR_UNSUPPORTED, "query heads per kv head %d unsupported (6, 8, 16)", QG);
  if (max_num_kv_splits < 1 || max_num_kv_splits > 256)
    return fail(UQ_ERR_INVALID_ARG, "max_num_kv_splits %d outside [1, 256]", max_num_kv_splits);
  if (num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(UQ_ERR_INVALID_ARG, "num_blocks %d / max_blocks_per_seq %d must be >= 1", num_blocks, max_blocks_per_seq);
  if ((int64_t)num_blocks * block_size >= ((int64_t)1 << 31) ||
      (int64_t)max_blocks_per_seq * block_size >= ((int64_t)1 << 31))
    return fail(UQ_ERR_INVALID_ARG, "num_blocks and max_blocks_per_seq times block_size must be < 2^31");
  if (B > 65535) return fail(UQ_ERR_INVALID_ARG, "B %d exceeds 65535", B);
  if (Hk > 256) return fail(UQ_ERR_UNSUPPORTED, "Hk %d exceeds 256", Hk);
  if ((int64_t)B * Hq * max_num_kv_splits > ((int64_t)1 << 30))
    return fail(UQ_ERR_INVALID_ARG, "B * Hq * max_num_kv_splits exceeds 2^30");
  if (!(scale == scale)) return fail(UQ_ERR_INVALID_ARG, "scale is NaN");
  if (B == 0) {
    *noop = true;
    return UQ_OK;
  }
  if (!query || !kv_cache || !block_table || !workspace || !out)
    return fail(UQ_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(query, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(workspace, 16))
    return fail(UQ_ERR_INVALID_ARG, "query, kv_cache, workspace and out must be 16-byte aligned");
  if (!aligned(block_table, 4))
    return fail(UQ_ERR_INVALID_ARG, "block_table must be 4-byte aligned");
  if (q_stride_head < head_dim || q_stride_seq < (int64_t)(Hq - 1) * q_stride_head + head_dim ||
      q_stride_head % 8 || q_stride_seq % 8)
    return fail(UQ_ERR_INVALID_ARG, "query strides (%lld, %lld) must cover a [Hq][256] row and be multiples of 8",
                (long long)q_stride_seq, (long long)q_stride_head);
  const size_t need = uq_decode_workspace_bytes(B, Hq, head_dim, max_num_kv_splits);
  if (workspace_bytes < need)
    return fail(UQ_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  return UQ_OK;
}

uq_status launch_checked_decode(const void* query, const void* kv_cache, const int32_t* block_table,
                                const uq::SeqRows& rows, float scale, const float* sinks,
                                int max_num_kv_splits,
                                void* workspace, void* out, int B, int Hq, int Hk, int num_blocks,
                                int max_blocks_per_seq, int64_t q_stride_seq, int64_t q_stride_head,
                                void* stream) {
  unsigned int* err = nullptr;
  uq_status st = error_word(&err);
  if (st != UQ_OK) return st;
  cudaError_t e = uq::launch_decode(static_cast<const uint16_t*>(query), q_stride_seq, q_stride_head,
                                    static_cast<const uint8_t*>(kv_cache), block_table, rows, scale,
                                    sinks, B, Hq, Hk, num_blocks, max_blocks_per_seq, max_num_kv_splits,
                                    workspace, static_cast<uint16_t*>(out), err,
                                    static_cast<cudaStream_t>(stream), g_ev_before_stage1,
                                    g_ev_after_stage1);
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

uq_status uq_decode_ex(const void* query, const void* kv_cache, const int32_t* block_table,
                       const int32_t* seq_lens, float scale, const float* sinks, int sliding_window,
                       int max_num_kv_splits, void* workspace, size_t workspace_bytes, void* out,
                       int B, int Hq, int Hk, int head_dim, int num_blocks, int block_size,
                       int max_blocks_per_seq, int slot_bytes, int64_t q_stride_seq,
                       int64_t q_stride_head, void* stream) {
  bool noop = false;
  uq_status st = check_decode(query, kv_cache, block_table, scale, max_num_kv_splits, workspace,
                              workspace_bytes, out, B, Hq, Hk, head_dim, num_blocks, block_size,
                              max_blocks_per_seq, slot_bytes, q_stride_seq, q_stride_head, &noop);
  if (st != UQ_OK) return st;
  if (noop) return ok();
  if (!seq_lens) return fail(UQ_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(seq_lens, 4) || (sinks && !aligned(sinks, 4)))
    return fail(UQ_ERR_INVALID_ARG, "block_table, seq_lens and sinks must be 4-byte aligned");
  const uq::SeqRows rows{seq_lens, (int64_t)max_blocks_per_seq, -1, sliding_window,
                         log2_tiles_per_page(block_size), max_blocks_per_seq * (block_size / 16), 1, B};
  return launch_checked_decode(query, kv_cache, block_table, rows, scale, sinks, max_num_kv_splits,
                               workspace, out, B, Hq, Hk, num_blocks, max_blocks_per_seq,
                               q_stride_seq, q_stride_head, stream);
}

uq_status uq_decode(const void* query, const void* kv_cache, const int32_t* block_table,
                    const int32_t* seq_lens, float scale, int max_num_kv_splits, void* workspace,
                    size_t workspace_bytes, void* out, int B, int Hq, int Hk, int head_dim,
                    int num_blocks, int block_size, int max_blocks_per_seq, int slot_bytes,
                    int64_t q_stride_seq, int64_t q_stride_head, void* stream) {
  return uq_decode_ex(query, kv_cache, block_table, seq_lens, scale, nullptr, 0, max_num_kv_splits,
                      workspace, workspace_bytes, out, B, Hq, Hk, head_dim, num_blocks, block_size,
                      max_blocks_per_seq, slot_bytes, q_stride_seq, q_stride_head, stream);
}

uq_status uq_decode_multi_query(const void* query, const void* kv_cache, const int32_t* block_table,
                                int cached_len, int q_len, float scale, const float* sinks,
                                int sliding_window, int max_num_kv_splits,
                                void* workspace, size_t workspace_bytes, void* out, int Hq, int Hk,
                                int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
                                int slot_bytes, int64_t q_stride_tok, int64_t q_stride_head,
                                void* stream) {
  if (cached_len < 0) return fail(UQ_ERR_INVALID_ARG, "cached_len %d < 0", cached_len);
  bool noop = false;
  uq_status st = check_decode(query, kv_cache, block_table, scale, max_num_kv_splits, workspace,
                              workspace_bytes, out, q_len, Hq, Hk, head_dim, num_blocks, block_size,
                              max_blocks_per_seq, slot_bytes, q_stride_tok, q_stride_head, &noop);
  if (st != UQ_OK) return st;
  if (noop) return ok();
  if ((int64_t)cached_len + q_len > (int64_t)max_blocks_per_seq * block_size)
    return fail(UQ_ERR_INVALID_ARG, "cached_len %d + q_len %d exceeds the %d pages of block_table",
                cached_len, q_len, max_blocks_per_seq);
  if (sinks && !aligned(sinks, 4)) return fail(UQ_ERR_INVALID_ARG, "sinks must be 4-byte aligned");
  // Two consecutive chunk positions share a work unit when that makes at most
  // 16 query rows (6 or 8 query heads per kv head): each page is read and
  // dequantised once for both.
  const int pack = (q_len > 1 && 2 * (Hq / Hk) <= 16) ? 2 : 1;
  const uq::SeqRows rows{nullptr, 0, cached_len, sliding_window, log2_tiles_per_page(block_size),
                         max_blocks_per_seq * (block_size / 16), pack, q_len};
  return launch_checked_decode(query, kv_cache, block_table, rows, scale, sinks, max_num_kv_splits,
                               workspace, out, q_len, Hq, Hk, num_blocks, max_blocks_per_seq,
                               q_stride_tok, q_stride_head, stream);
}

uq_status uq_check_device_error(void* stream, unsigned int* flags_out) {
  unsigned int* err = nullptr;
  uq_status st = error_word(&err);
  if (st != UQ_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int flags = 0;
  e = cudaMemcpyFromSymbol(&flags, g_device_error_word, sizeof flags);
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof zero);
  if (e != cudaSuccess) return fail(UQ_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(e));
  if (flags_out) *flags_out = flags;
  if (flags) return fail(UQ_ERR_DEVICE_FLAG, "device error word 0x%x", flags);
  return ok();
}

}  // extern "C"
