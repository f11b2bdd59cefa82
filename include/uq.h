/*
 * uq.h -- C ABI of the UltraQuant 4-bit KV-cache library for NVIDIA GB300
 * (sm_103a): paged store into an FP4 E2M1 + UE8M0 cache with a Hadamard-
 * rotated K, and split-KV paged decode attention over that cache.
 *
 * Sources (vLLM API documentation pages):
 *   vllm.v1.attention.backends.ultraquant_attn, UltraQuantAttentionImpl
 *     (class docstring: "FP4 E2M1 + UE8M0, rotated K"; _ensure_on_device:
 *     the Hadamard rotation; _store_kv: the store seam; _decode_attention:
 *     the decode seam and its workspace)
 *   vllm.v1.attention.ops.flydsl_ultraquant_decode
 *     (flydsl_ultraquant_decode_attention: query prologue with the E4M3
 *     haircut, stage-1 launch, partition reduce; _fp4_value_lut)
 *   vllm.v1.attention.ops.turboquant_soa.triton_turboquant_decode_v2
 *     (triton_turboquant_decode_attention_v2: fixed split count for graph
 *     capture, split partials and their combine)
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller.  The
 *     library allocates no memory and never synchronises inside its compute
 *     calls (uq_store, uq_store_rotated_f32, uq_decode, uq_decode_ex,
 *     uq_decode_multi_query, uq_full_dequant); work is enqueued on `stream`
 *     (a cudaStream_t passed as void*; NULL is the legacy default stream).
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call returns an error code and enqueues nothing.  The message
 *     of the last error on the calling thread is in uq_last_error().
 *   - Index errors that only the device can see (a page id outside
 *     [0, num_blocks), a slot beyond the cache) never fault: the affected
 *     token is skipped and a bit is set in a device error word that
 *     uq_check_device_error() reads.
 *   - Supported shapes: head_dim D = 256, query heads per KV head (Hq / Hk)
 *     in {6, 8, 16}, block_size in {16, 32, 64, 128, 256} for decode and
 *     dequantisation (any block_size >= 1 for the store); other values
 *     return UQ_ERR_UNSUPPORTED.  Kernels walk pages in 16-token tiles.
 *
 * Cache layout (the pages give only kv_cache's shape, (num_blocks,
 * block_size, Hk, slot_size) uint8; the byte layout below is this library's)
 *   Slot of (page p, offset o, kv head h) starts at byte
 *   ((p * block_size + o) * Hk + h) * slot_bytes, slot_bytes = 272 for D = 256:
 *     [  0,128) K codes: element 2j in the low nibble of byte j, 2j+1 high
 *     [128,256) V codes, same packing
 *     [256,264) K block-scale bytes, one UE8M0 per 32 consecutive elements
 *     [264,272) V block-scale bytes
 *   A code c decodes to E2M1(c) * 2^(byte - 127), E2M1 codes 0..7 being
 *   +{0, .5, 1, 1.5, 2, 3, 4, 6} and 8..15 their negatives.  K is stored
 *   rotated: k_rot = k H with H[i][j] = (-1)^popcount(i&j) / 16.  V is not
 *   rotated.
 */
#ifndef UQ_H
#define UQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    UQ_OK = 0,
    UQ_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad size or stride */
    UQ_ERR_UNSUPPORTED = 2,          /* a shape outside the supported set */
    UQ_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < uq_decode_workspace_bytes() */
    UQ_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed */
    UQ_ERR_DEVICE_FLAG = 5           /* the device error word was non-zero */
} uq_status;

/* Device error word bits (uq_check_device_error). */
#define UQ_DEVERR_BAD_PAGE 1u        /* block_table entry outside [0, num_blocks) */
#define UQ_DEVERR_BAD_SLOT 2u        /* slot_mapping entry >= num_blocks * block_size */
#define UQ_DEVERR_TIMEOUT  4u        /* a bounded wait on an async copy gave up */

/* Library version, major * 10000 + minor * 100 + patch. */
int uq_version(void);

/* Bytes of one (token, kv head) slot for head_dim: D + D/16 (272 for D = 256).
 * Returns 0 for an unsupported head_dim. */
size_t uq_slot_bytes(int head_dim);

/*
 * Workspace bytes uq_decode needs for a batch of up to B sequences with Hq
 * query heads and max_num_kv_splits splits: per (sequence, query head,
 * split) the split's partial output (256 fp32), its log-sum-exp (fp32) and
 * one 4-byte work-list entry, plus 12 bytes per sequence and a 64-byte
 * header, i.e. B * Hq * S * 1032 + 12 * B + 64, rounded up to 256 bytes.  It
 * depends only on its arguments, so a caller can size the workspace once for
 * its largest batch before capturing a CUDA graph (the reference pre-grows
 * its pool before capture for the same reason, _ensure_on_device and
 * _SegmBufPool).  Returns 0 for invalid arguments (B < 1, Hq < 1, head_dim
 * != 256, S outside [1, 256]).
 */
size_t uq_decode_workspace_bytes(int B, int Hq, int head_dim, int max_num_kv_splits);

/*
 * uq_store -- rotate K by the Hadamard matrix and pack K and V into the
 * paged FP4 cache (ultraquant_attn, UltraQuantAttentionImpl._store_kv).
 *
 *   key, value    bf16, element (n, h, d) at n * key_stride_tok + h * D + d
 *                 (value_stride_tok for value); 16-byte aligned, strides in
 *                 elements and multiples of 8.
 *   kv_cache      uint8 [num_blocks][block_size][Hk][slot_bytes], written.
 *   slot_mapping  int64 [num_tokens]; token n goes to slot slot_mapping[n]
 *                 (page = slot / block_size, offset = slot % block_size).
 *                 A negative slot skips the token; a slot >= num_blocks *
 *                 block_size skips it and sets UQ_DEVERR_BAD_SLOT.  A
 *                 skipped token's K and V rows are still read (they must
 *                 be valid memory like every other row); only its slot is
 *                 not written.
 *
 * Per (token, head): K is converted to fp32 (exact), transformed by the
 * unnormalised fast Walsh-Hadamard butterfly in the fixed stage order
 * h = 1, 2, ..., 128 (pair (i, i+h) -> (a+b, a-b)) and multiplied by 1/16.
 * Each 32-element block of rotated K and of V gets the UE8M0 byte
 * max(0, biased_exponent(amax) - 2) (shared exponent floor(log2 amax) - 2,
 * clamped at -127) and E2M1 codes of x * 2^-(byte-127), rounded to nearest
 * even with saturation at +-6; a negative value that rounds to zero keeps
 * its sign bit.  num_tokens == 0 is a no-op.
 */
uq_status uq_store(const void *key, const void *value, void *kv_cache,
                   const int64_t *slot_mapping, int64_t num_tokens,
                   int num_kv_heads, int head_dim, int num_blocks, int block_size,
                   int slot_bytes, int64_t key_stride_tok, int64_t value_stride_tok,
                   void *stream);

/*
 * uq_store_rotated_f32 -- the quantise-and-pack half of uq_store for K that
 * is already rotated: key_rot and value are fp32, contiguous
 * [num_tokens][Hk][D], 16-byte aligned.  Same slot rules, scale rule and
 * rounding as uq_store, without the rotation.  It lets a caller check the
 * packed bytes against another implementation that quantises the same fp32
 * rotated K.
 */
uq_status uq_store_rotated_f32(const float *key_rot, const float *value,
                               void *kv_cache, const int64_t *slot_mapping,
                               int64_t num_tokens, int num_kv_heads, int head_dim,
                               int num_blocks, int block_size, int slot_bytes,
                               void *stream);

/*
 * uq_decode -- split-KV paged decode attention over the FP4 cache
 * (ultraquant_attn, UltraQuantAttentionImpl._decode_attention;
 * flydsl_ultraquant_decode, flydsl_ultraquant_decode_attention).
 *
 *   query        bf16, element (b, r, d) at b * q_stride_seq +
 *                r * q_stride_head + d (elements; 16-byte aligned rows).
 *   kv_cache     uint8 cache written by uq_store (read only).
 *   block_table  int32 [B][max_blocks_per_seq]: page ids of each sequence.
 *   seq_lens     int32 [B]: tokens of each sequence, 0 <= L <=
 *                max_blocks_per_seq * block_size (larger values are clamped
 *                to that capacity on the device).
 *   scale        softmax scale applied to q'.k (typically 1/sqrt(D)).
 *   max_num_kv_splits  S, the fixed number of splits per (sequence, kv head);
 *                1 <= S <= 256.  The grid depends only on (S, Hk, B), so the
 *                call can be captured once in a CUDA graph and replayed with
 *                new seq_lens / block_table contents.
 *   workspace    device scratch of at least
 *                uq_decode_workspace_bytes(B, Hq, D, S) bytes, 256-byte
 *                aligned; contents need no initialisation.
 *   out          bf16 [B][Hq][D] contiguous, written.
 *
 * Per query head r (kv head r / (Hq/Hk)): q' = bf16(e4m3(fp32(q) H)) (the
 * E4M3 "haircut", round to nearest even, saturating); s_t = scale * q'.k_t
 * over the L tokens of the sequence, k_t the dequantised rotated K;
 * out = softmax(s) . V (dequantised), rounded to bf16.  A sequence with
 * L == 0 gets out = 0.  Supported Hk <= 256, B <= 65535.  Four kernels run
 * on the stream: a one-CTA plan that divides every sequence into up to S
 * splits of whole pages (the split size is chosen on the device from the
 * batch's total length, so the work list has a few units per resident CTA)
 * and orders the units longest first; the split-KV kernel (persistent CTAs
 * taking units from that list); an exact fp32 pass over the units that hold
 * a token whose K block scales span 2^28 or more (the split-KV kernel keeps
 * K block scales relative to each token's largest one in f16 and lists such
 * units instead; with no such token the pass returns at once); and the merge
 * of each row's splits.  V blocks 2^28 or more below their token's largest
 * V block are dropped by the split-KV kernel (each such value is below
 * 6 * 2^-28 of that block in magnitude).
 */
uq_status uq_decode(const void *query, const void *kv_cache,
                    const int32_t *block_table, const int32_t *seq_lens,
                    float scale, int max_num_kv_splits, void *workspace,
                    size_t workspace_bytes, void *out, int B, int Hq, int Hk,
                    int head_dim, int num_blocks, int block_size,
                    int max_blocks_per_seq, int slot_bytes, int64_t q_stride_seq,
                    int64_t q_stride_head, void *stream);

/*
 * uq_decode_ex -- uq_decode with attention sinks and a sliding window
 * (ultraquant_attn, UltraQuantAttentionImpl: sinks and sliding_window, which
 * the backend hands to its unified attention with window_size =
 * (sliding_window - 1, 0); the FlyDSL kernel rejects both).
 *
 *   sinks           fp32 [Hq] device array of sink logits, or NULL.  Query
 *                   head r's softmax becomes e^(s_t - m) / (e^(z_r - m) +
 *                   sum_t e^(s_t - m)): the sink z_r (same units as
 *                   scale * q'.k, finite or -inf) joins the denominator only.
 *   sliding_window  W > 0: a row of length L attends to tokens
 *                   [max(0, L - W), L) only; W <= 0: no window.
 *
 * Everything else as uq_decode, which is uq_decode_ex(..., NULL, 0, ...).
 * The window moves the pages a row reads, so the work list (and the time)
 * shrinks with it.
 */
uq_status uq_decode_ex(const void *query, const void *kv_cache,
                       const int32_t *block_table, const int32_t *seq_lens,
                       float scale, const float *sinks, int sliding_window,
                       int max_num_kv_splits, void *workspace, size_t workspace_bytes,
                       void *out, int B, int Hq, int Hk, int head_dim, int num_blocks,
                       int block_size, int max_blocks_per_seq, int slot_bytes,
                       int64_t q_stride_seq, int64_t q_stride_head, void *stream);

/*
 * uq_decode_multi_query -- attention of a short continuation chunk (or of
 * the draft tokens of speculative decoding) over the FP4 cache
 * (ultraquant_attn, UltraQuantAttentionImpl._prefill_attention, continuation
 * chunks with q_len <= _CONTINUATION_DECODE_THRESHOLD: the decode-shaped
 * kernel run on synthetic seq_lens = arange(cached_len + 1, seq_len + 1) and
 * the sequence's block-table row expanded q_len times).
 *
 *   query        bf16, row i of the chunk (its token at absolute position
 *                cached_len + i) and query head r at i * q_stride_tok +
 *                r * q_stride_head + d.
 *   kv_cache     uint8 cache that already holds the sequence's first
 *                cached_len + q_len tokens, the chunk's own K/V included
 *                (written by uq_store before the call).
 *   block_table  int32 [max_blocks_per_seq]: the one sequence's page ids.
 *   workspace    uq_decode_workspace_bytes(q_len, Hq, D, S) bytes.
 *   out          bf16 [q_len][Hq][D] contiguous, written.
 *
 * Row i attends causally to tokens 0 .. cached_len + i: exactly uq_decode
 * on a batch of q_len rows with seq_lens[i] = cached_len + i + 1 that all
 * read the same pages, without materialising those arrays.  With 6 or 8
 * query heads per KV head two consecutive rows share each work unit, so a
 * page is read and dequantised once per pair of rows; the pairs' units run
 * side by side, so HBM reads each page about once.  Results equal uq_decode
 * on that batch within the decode tolerance, not bit for bit.
 * sinks and sliding_window as in uq_decode_ex; the window counts back from
 * each row's own position.  Requires cached_len >= 0 and cached_len + q_len
 * <= max_blocks_per_seq * block_size; q_len == 0 is a no-op.  Other rules as
 * uq_decode.
 */
uq_status uq_decode_multi_query(const void *query, const void *kv_cache,
                                const int32_t *block_table, int cached_len, int q_len,
                                float scale, const float *sinks, int sliding_window,
                                int max_num_kv_splits, void *workspace,
                                size_t workspace_bytes, void *out, int Hq, int Hk,
                                int head_dim, int num_blocks, int block_size,
                                int max_blocks_per_seq, int slot_bytes,
                                int64_t q_stride_tok, int64_t q_stride_head, void *stream);

/*
 * uq_full_dequant -- expand one sequence's cached prefix to bf16
 * (ultraquant_attn, UltraQuantAttentionImpl._ultraquant_continuation_prefill:
 * the call to ultraquant_full_dequant_kv that feeds a large continuation
 * chunk's dense prefill).
 *
 *   kv_cache     uint8 cache written by uq_store (read only).
 *   block_table  int32 [n_pages]: the sequence's page ids, in order.
 *   n_pages      pages to expand (>= 0): alloc_len = n_pages * block_size
 *                rows, ceil(cached_len / block_size) pages for a prefix of
 *                cached_len tokens.
 *   k_out, v_out bf16 [Hk][alloc_len][D] contiguous (the pages' buffer
 *                (1, Hk, alloc_len, D) without the leading 1), written;
 *                16-byte aligned.  Row t of page p is row p * block_size + t.
 *
 * K stays Hadamard-rotated, as stored; V is in the original space.  Every
 * element is E2M1(code) * 2^(byte - 127) rounded to bf16 (exact: at most two
 * significant bits; a product beyond bf16's range becomes +-inf, which the
 * store never produces).  A page id outside [0, num_blocks) writes zero rows
 * and sets UQ_DEVERR_BAD_PAGE.  n_pages == 0 is a no-op.  Supported:
 * head_dim 256, block_size in {16, 32, 64, 128, 256}, 1 <= Hk <= 256,
 * n_pages * block_size < 2^31 and n_pages * (block_size / 16) * Hk < 2^31.
 */
uq_status uq_full_dequant(const void *kv_cache, const int32_t *block_table, int n_pages,
                          void *k_out, void *v_out, int Hk, int head_dim, int num_blocks,
                          int block_size, int slot_bytes, void *stream);

/*
 * uq_decode_static_scratch -- uq_decode for callers that cannot allocate
 * device memory.  The paper has no counterpart; this entry point exists for
 * integrations where nobody can hand uq_decode a workspace: for example a
 * plugin whose enqueue step must not call cudaMalloc (the call can
 * synchronise the device and can fail in the middle of serving), or a host
 * that keeps all device memory in its own pool and gives its kernels no
 * allocator.  It runs exactly uq_decode, with the split partials in a scratch
 * array of 32 MiB that the library declares statically: every GPU that loads
 * this library holds that array until the process exits.
 *
 * Arguments are those of uq_decode without workspace and workspace_bytes.
 * A batch whose uq_decode_workspace_bytes(B, Hq, 256, max_num_kv_splits)
 * exceeds 32 MiB (roughly B * Hq * max_num_kv_splits > 32480) is rejected
 * with UQ_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  The call allocates
 * nothing.  The first call on a device (and the first after its CUDA
 * context changes, e.g. after a device reset) looks up the array's device
 * address; make that first call before any stream capture.  All calls on a device
 * share the one array, and it keeps the previous call's partials (nothing in
 * it needs to start at zero), so calls that can overlap on the GPU (for
 * example on two streams without an ordering between them) race.
 */
uq_status uq_decode_static_scratch(const void *query, const void *kv_cache,
                                   const int32_t *block_table, const int32_t *seq_lens,
                                   float scale, int max_num_kv_splits, void *out, int B,
                                   int Hq, int Hk, int head_dim, int num_blocks,
                                   int block_size, int max_blocks_per_seq, int slot_bytes,
                                   int64_t q_stride_seq, int64_t q_stride_head,
                                   void *stream);

/*
 * Profiling hook.  When set (non-NULL), the next uq_decode calls made by the
 * calling thread record `before_stage1` on their stream just before the
 * stage-1 kernel and `after_stage1` just after it, so a caller can time the
 * split-KV kernel alone with cudaEventElapsedTime.  Both are cudaEvent_t
 * handles passed as void*, owned by the caller; NULL, NULL turns it off.
 * Recording is part of the enqueued work, so it is captured into a CUDA
 * graph like the kernels.  Always returns UQ_OK.
 */
uq_status uq_set_timing_events(void *before_stage1, void *after_stage1);

/* Message describing the last error returned on the calling thread ("" if none). */
const char *uq_last_error(void);

/*
 * Synchronise `stream`, read and clear the device error word of the current
 * device.  Returns UQ_OK if no bit was set, UQ_ERR_DEVICE_FLAG (bits in
 * *flags_out when non-NULL) if any was, UQ_ERR_CUDA on a runtime error.
 * Intended for tests and debugging, outside the hot path.
 */
uq_status uq_check_device_error(void *stream, unsigned int *flags_out);

#ifdef __cplusplus
}
#endif

#endif /* UQ_H */
