// uq_noalloc.cu -- uq_decode for callers that cannot allocate device memory.
//
// uq_decode needs a workspace for its split partials, and the caller owns it.
// Some callers have no way to provide one.  Examples: a plugin whose enqueue
// step must not call cudaMalloc, because that call can synchronise the
// device and can fail in the middle of serving; a host that hands all device
// memory to its own pool and gives its kernels no allocator; code that is
// only allowed to pass the tensors it was given.  uq_decode_static_scratch
// uses instead a fixed scratch array that the library owns, declared below.
// Every GPU that loads this library holds the array until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "uq.h"

namespace uq {
uq_status set_error(uq_status code, const char* msg);
cudaError_t current_context_id(unsigned long long* id);
}

namespace {

// Upper bound of uq_decode_workspace_bytes(B, Hq, 256, S) that the static
// scratch can serve: 32 MiB, roughly B * Hq * S <= 32480.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress, once per device and
// CUDA context (after a device reset the array lives at a new address).
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

void* g_scratch_dev_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};
std::mutex g_scratch_mutex;

}  // namespace

extern "C" uq_status uq_decode_static_scratch(
    const void* query, const void* kv_cache, const int32_t* block_table,
    const int32_t* seq_lens, float scale, int max_num_kv_splits, void* out, int B, int Hq,
    int Hk, int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
    int slot_bytes, int64_t q_stride_seq, int64_t q_stride_head, void* stream) {
  const size_t need = uq_decode_workspace_bytes(B, Hq, head_dim, max_num_kv_splits);
  if (B > 0 && need > kStaticScratchBytes)
    return uq::set_error(UQ_ERR_WORKSPACE_TOO_SMALL,
                         "uq_decode_static_scratch: this batch needs more scratch than the "
                         "library's fixed 32 MiB (roughly B * Hq * max_num_kv_splits <= 32480); "
                         "use uq_decode with a caller-provided workspace");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return uq::set_error(UQ_ERR_CUDA, "uq_decode_static_scratch: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return uq::set_error(UQ_ERR_UNSUPPORTED, "uq_decode_static_scratch: device index out of range");
  unsigned long long ctx = 0;
  if (uq::current_context_id(&ctx) != cudaSuccess)
    return uq::set_error(UQ_ERR_CUDA, "uq_decode_static_scratch: no current CUDA context");
  void* scratch = nullptr;
  {
    // First call on a device (or in a new context of it): look up the device
    // address of the array with that device current.
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_dev_ptr[dev] || g_scratch_ctx[dev] != ctx) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess || !p)
        return uq::set_error(UQ_ERR_CUDA, "uq_decode_static_scratch: cudaGetSymbolAddress failed");
      g_scratch_dev_ptr[dev] = p;
      g_scratch_ctx[dev] = ctx;
    }
    scratch = g_scratch_dev_ptr[dev];
  }
  return uq_decode(query, kv_cache, block_table, seq_lens, scale, max_num_kv_splits, scratch,
                   kStaticScratchBytes, out, B, Hq, Hk, head_dim, num_blocks, block_size,
                   max_blocks_per_seq, slot_bytes, q_stride_seq, q_stride_head, stream);
}
