"""ctypes binding of libuq.so: the C ABI of include/uq.h under the same names.

Argument marshalling only: each function checks shapes and dtypes of the
torch tensors it is given, passes their device pointers, sizes and strides
to the C entry point, and raises ``UQError`` on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; there is no
other code path.  The library is loaded from the package's ``_build``
directory and the import fails loudly if it is missing or stale.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libuq.so")

UQ_OK = 0
UQ_ERR_INVALID_ARG = 1
UQ_ERR_UNSUPPORTED = 2
UQ_ERR_WORKSPACE_TOO_SMALL = 3
UQ_ERR_CUDA = 4
UQ_ERR_DEVICE_FLAG = 5

UQ_DEVERR_BAD_PAGE = 1
UQ_DEVERR_BAD_SLOT = 2
UQ_DEVERR_TIMEOUT = 4

HEAD_DIM = 256
SLOT_BYTES = 272

EXPORTED = ("uq_version", "uq_slot_bytes", "uq_decode_workspace_bytes", "uq_store",
            "uq_store_rotated_f32", "uq_decode", "uq_decode_ex", "uq_decode_multi_query",
            "uq_full_dequant",
            "uq_decode_static_scratch",
            "uq_set_timing_events", "uq_last_error", "uq_check_device_error")


class UQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"uq status {status}: {message}")
        self.status = status


_LIB = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libuq.so (raises OSError if it has not been built)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError(f"{p} not found: build it with bit_quantized_kv_gb300.build.build()")
    L = ctypes.CDLL(p)
    c_int, c_i64, c_sz, c_p, c_f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
    L.uq_version.restype = c_int
    L.uq_version.argtypes = []
    L.uq_slot_bytes.restype = c_sz
    L.uq_slot_bytes.argtypes = [c_int]
    L.uq_decode_workspace_bytes.restype = c_sz
    L.uq_decode_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int]
    L.uq_store.restype = c_int
    L.uq_store.argtypes = [c_p, c_p, c_p, c_p, c_i64, c_int, c_int, c_int, c_int, c_int,
                           c_i64, c_i64, c_p]
    L.uq_store_rotated_f32.restype = c_int
    L.uq_store_rotated_f32.argtypes = [c_p, c_p, c_p, c_p, c_i64, c_int, c_int, c_int, c_int,
                                       c_int, c_p]
    L.uq_decode.restype = c_int
    L.uq_decode.argtypes = [c_p, c_p, c_p, c_p, c_f, c_int, c_p, c_sz, c_p, c_int, c_int,
                            c_int, c_int, c_int, c_int, c_int, c_int, c_i64, c_i64, c_p]
    L.uq_decode_multi_query.restype = c_int
    L.uq_decode_multi_query.argtypes = [c_p, c_p, c_p, c_int, c_int, c_f, c_p, c_int, c_int, c_p,
                                        c_sz, c_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                        c_i64, c_i64, c_p]
    L.uq_decode_ex.restype = c_int
    L.uq_decode_ex.argtypes = [c_p, c_p, c_p, c_p, c_f, c_p, c_int, c_int, c_p, c_sz, c_p, c_int,
                               c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_i64, c_i64, c_p]
    L.uq_full_dequant.restype = c_int
    L.uq_full_dequant.argtypes = [c_p, c_p, c_int, c_p, c_p, c_int, c_int, c_int, c_int, c_int, c_p]
    L.uq_decode_static_scratch.restype = c_int
    L.uq_decode_static_scratch.argtypes = [c_p, c_p, c_p, c_p, c_f, c_int, c_p, c_int, c_int,
                                           c_int, c_int, c_int, c_int, c_int, c_int, c_i64,
                                           c_i64, c_p]
    L.uq_set_timing_events.restype = c_int
    L.uq_set_timing_events.argtypes = [c_p, c_p]
    L.uq_last_error.restype = ctypes.c_char_p
    L.uq_last_error.argtypes = []
    L.uq_check_device_error.restype = c_int
    L.uq_check_device_error.argtypes = [c_p, ctypes.POINTER(ctypes.c_uint)]
    if path is None:
        _LIB = L
    return L


def _check(status: int) -> None:
    if status != UQ_OK:
        raise UQError(status, load().uq_last_error().decode())


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    """dtype and rank of a tensor argument (the device is checked by _on_gpu,
    after the shape checks, so that those are visible without a GPU)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _on_gpu(**tensors) -> None:
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _decode_batch_args(query, kv_cache, block_table, seq_lens, out):
    """Checks shared by the batch decode wrappers, in the order a caller would
    fix them: dtypes and ranks, the query/out/cache layout, the block-table
    and length rows, then the device.  Returns (B, Hq, D, nb, bs, Hk, sb)."""
    _need(query, "query", torch.bfloat16, 3)
    _need(kv_cache, "kv_cache", torch.uint8, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    B, Hq, D = query.shape
    if query.stride(2) != 1:
        raise ValueError("query rows must be contiguous along the head dim")
    if out.shape != query.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like query")
    if not (kv_cache.is_contiguous() and block_table.is_contiguous() and seq_lens.is_contiguous()):
        raise ValueError("kv_cache, block_table and seq_lens must be contiguous")
    if block_table.shape[0] < B or seq_lens.shape[0] < B:
        raise ValueError("block_table / seq_lens have fewer rows than the batch")
    _on_gpu(query=query, kv_cache=kv_cache, block_table=block_table, seq_lens=seq_lens, out=out)
    nb, bs, Hk, sb = kv_cache.shape
    return B, Hq, D, nb, bs, Hk, sb


def uq_version() -> int:
    return load().uq_version()


def uq_slot_bytes(head_dim: int = HEAD_DIM) -> int:
    return load().uq_slot_bytes(head_dim)


def uq_decode_workspace_bytes(B: int, Hq: int, head_dim: int, max_num_kv_splits: int) -> int:
    return load().uq_decode_workspace_bytes(B, Hq, head_dim, max_num_kv_splits)


def uq_last_error() -> str:
    return load().uq_last_error().decode()


def uq_store(key: torch.Tensor, value: torch.Tensor, kv_cache: torch.Tensor,
             slot_mapping: torch.Tensor, stream=None) -> None:
    """key, value bf16 [N, Hk, D] (rows may be strided); kv_cache uint8
    [num_blocks, block_size, Hk, 272]; slot_mapping int64 [N]."""
    _need(key, "key", torch.bfloat16, 3)
    _need(value, "value", torch.bfloat16, 3)
    _need(kv_cache, "kv_cache", torch.uint8, 4)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    N, Hk, D = key.shape
    if value.shape != key.shape or slot_mapping.shape[0] != N:
        raise ValueError("key/value/slot_mapping shapes disagree")
    if key.stride(2) != 1 or key.stride(1) != D or value.stride(2) != 1 or value.stride(1) != D:
        raise ValueError("key/value must be contiguous within a token row")
    if not kv_cache.is_contiguous() or not slot_mapping.is_contiguous():
        raise ValueError("kv_cache and slot_mapping must be contiguous")
    nb, bs, hk2, sb = kv_cache.shape
    if hk2 != Hk:
        raise ValueError("kv_cache head count differs from key")
    _on_gpu(key=key, value=value, kv_cache=kv_cache, slot_mapping=slot_mapping)
    _check(load().uq_store(key.data_ptr(), value.data_ptr(), kv_cache.data_ptr(),
                           slot_mapping.data_ptr(), N, Hk, D, nb, bs, sb,
                           key.stride(0), value.stride(0), _stream_ptr(stream)))


def uq_store_rotated_f32(key_rot: torch.Tensor, value: torch.Tensor, kv_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, stream=None) -> None:
    """key_rot (already rotated) and value fp32 contiguous [N, Hk, D]."""
    _need(key_rot, "key_rot", torch.float32, 3)
    _need(value, "value", torch.float32, 3)
    _need(kv_cache, "kv_cache", torch.uint8, 4)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    if not (key_rot.is_contiguous() and value.is_contiguous() and kv_cache.is_contiguous()
            and slot_mapping.is_contiguous()):
        raise ValueError("uq_store_rotated_f32 needs contiguous tensors")
    _on_gpu(key_rot=key_rot, value=value, kv_cache=kv_cache, slot_mapping=slot_mapping)
    N, Hk, D = key_rot.shape
    nb, bs, _, sb = kv_cache.shape
    _check(load().uq_store_rotated_f32(key_rot.data_ptr(), value.data_ptr(), kv_cache.data_ptr(),
                                       slot_mapping.data_ptr(), N, Hk, D, nb, bs, sb,
                                       _stream_ptr(stream)))


def uq_decode(query: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
              seq_lens: torch.Tensor, scale: float, max_num_kv_splits: int,
              workspace: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """query bf16 [B, Hq, D] (row-strided allowed); kv_cache uint8
    [num_blocks, 16, Hk, 272]; block_table int32 [B, max_blocks]; seq_lens
    int32 [B]; workspace uint8 (see uq_decode_workspace_bytes); out bf16
    [B, Hq, D] contiguous.  Returns ``out``."""
    B, Hq, D, nb, bs, Hk, sb = _decode_batch_args(query, kv_cache, block_table, seq_lens, out)
    _on_gpu(workspace=workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().uq_decode(query.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                            seq_lens.data_ptr(), float(scale), int(max_num_kv_splits),
                            workspace.data_ptr(), ws_bytes, out.data_ptr(), B, Hq, Hk, D,
                            nb, bs, block_table.shape[1], sb, query.stride(0), query.stride(1),
                            _stream_ptr(stream)))
    return out


def uq_decode_ex(query: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, scale: float, sinks: torch.Tensor | None,
                 sliding_window: int, max_num_kv_splits: int, workspace: torch.Tensor,
                 out: torch.Tensor, stream=None) -> torch.Tensor:
    """uq_decode with optional sink logits (fp32 [Hq] CUDA tensor or None)
    and a sliding window (> 0: the last ``sliding_window`` tokens)."""
    B, Hq, D, nb, bs, Hk, sb = _decode_batch_args(query, kv_cache, block_table, seq_lens, out)
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, 1)
        if sinks.shape[0] != Hq or not sinks.is_contiguous():
            raise ValueError("sinks must be a contiguous fp32 [Hq] tensor")
    _on_gpu(workspace=workspace, sinks=sinks)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().uq_decode_ex(query.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                               seq_lens.data_ptr(), float(scale),
                               None if sinks is None else sinks.data_ptr(), int(sliding_window),
                               int(max_num_kv_splits), workspace.data_ptr(), ws_bytes, out.data_ptr(),
                               B, Hq, Hk, D, nb, bs, block_table.shape[1], sb, query.stride(0),
                               query.stride(1), _stream_ptr(stream)))
    return out


def uq_decode_multi_query(query: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                          cached_len: int, scale: float, max_num_kv_splits: int,
                          workspace: torch.Tensor, out: torch.Tensor, stream=None,
                          sinks: torch.Tensor | None = None, sliding_window: int = 0) -> torch.Tensor:
    """query bf16 [q_len, Hq, D] (the chunk's rows, row-strided allowed);
    kv_cache uint8 [num_blocks, 16, Hk, 272] holding the first cached_len +
    q_len tokens; block_table int32 [max_blocks] (one sequence); workspace
    uint8 (uq_decode_workspace_bytes(q_len, ...)); out bf16 [q_len, Hq, D]
    contiguous.  Row i attends to tokens 0 .. cached_len + i.  Returns ``out``."""
    _need(query, "query", torch.bfloat16, 3)
    _need(kv_cache, "kv_cache", torch.uint8, 4)
    _need(block_table, "block_table", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    q_len, Hq, D = query.shape
    if query.stride(2) != 1:
        raise ValueError("query rows must be contiguous along the head dim")
    if out.shape != query.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like query")
    if not (kv_cache.is_contiguous() and block_table.is_contiguous()):
        raise ValueError("kv_cache and block_table must be contiguous")
    nb, bs, Hk, sb = kv_cache.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, 1)
        if sinks.shape[0] != Hq or not sinks.is_contiguous():
            raise ValueError("sinks must be a contiguous fp32 [Hq] tensor")
    _on_gpu(query=query, kv_cache=kv_cache, block_table=block_table, out=out, workspace=workspace,
            sinks=sinks)
    _check(load().uq_decode_multi_query(query.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                                        int(cached_len), q_len, float(scale),
                                        None if sinks is None else sinks.data_ptr(), int(sliding_window),
                                        int(max_num_kv_splits),
                                        workspace.data_ptr(), ws_bytes, out.data_ptr(), Hq, Hk, D, nb,
                                        bs, block_table.shape[0], sb, query.stride(0), query.stride(1),
                                        _stream_ptr(stream)))
    return out


def uq_full_dequant(kv_cache: torch.Tensor, block_table: torch.Tensor, k_out: torch.Tensor,
                    v_out: torch.Tensor, n_pages: int | None = None, stream=None):
    """Expand one sequence's pages to bf16: kv_cache uint8 [num_blocks, 16,
    Hk, 272]; block_table int32 [>= n_pages] page ids; k_out, v_out bf16
    [Hk, n_pages * 16, 256] contiguous (K stays rotated).  Returns (k_out, v_out)."""
    _need(kv_cache, "kv_cache", torch.uint8, 4)
    _need(block_table, "block_table", torch.int32, 1)
    _need(k_out, "k_out", torch.bfloat16, 3)
    _need(v_out, "v_out", torch.bfloat16, 3)
    n = block_table.shape[0] if n_pages is None else int(n_pages)
    nb, bs, Hk, sb = kv_cache.shape
    if n > block_table.shape[0]:
        raise ValueError("block_table has fewer entries than n_pages")
    for t in (k_out, v_out):
        if tuple(t.shape) != (Hk, n * bs, HEAD_DIM) or not t.is_contiguous():
            raise ValueError(f"k_out / v_out must be contiguous [{Hk}, {n * bs}, {HEAD_DIM}]")
    if not (kv_cache.is_contiguous() and block_table.is_contiguous()):
        raise ValueError("kv_cache and block_table must be contiguous")
    _on_gpu(kv_cache=kv_cache, block_table=block_table, k_out=k_out, v_out=v_out)
    _check(load().uq_full_dequant(kv_cache.data_ptr(), block_table.data_ptr(), n, k_out.data_ptr(),
                                  v_out.data_ptr(), Hk, HEAD_DIM, nb, bs, sb, _stream_ptr(stream)))
    return k_out, v_out


def uq_decode_static_scratch(query: torch.Tensor, kv_cache: torch.Tensor,
                             block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             max_num_kv_splits: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """uq_decode without a workspace argument, for callers that cannot
    allocate device memory: the split partials go to the library's fixed
    32 MiB scratch (roughly B * Hq * max_num_kv_splits <= 32480).  Calls that may run
    concurrently on the GPU share that scratch and must not overlap."""
    B, Hq, D, nb, bs, Hk, sb = _decode_batch_args(query, kv_cache, block_table, seq_lens, out)
    _check(load().uq_decode_static_scratch(query.data_ptr(), kv_cache.data_ptr(),
                                           block_table.data_ptr(), seq_lens.data_ptr(),
                                           float(scale), int(max_num_kv_splits), out.data_ptr(),
                                           B, Hq, Hk, D, nb, bs, block_table.shape[1], sb,
                                           query.stride(0), query.stride(1), _stream_ptr(stream)))
    return out


def uq_set_timing_events(before_stage1=None, after_stage1=None) -> None:
    """Record two torch.cuda.Event objects around decode stage 1 of the
    following uq_decode calls on this thread (None, None turns it off)."""
    def handle(ev):
        if ev is None:
            return None
        return ev.cuda_event or None
    _check(load().uq_set_timing_events(handle(before_stage1), handle(after_stage1)))


def uq_check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits.

    Raises UQError only for runtime failures; a set bit is returned, not
    raised, so callers can assert on it."""
    flags = ctypes.c_uint(0)
    st = load().uq_check_device_error(_stream_ptr(stream), ctypes.byref(flags))
    if st not in (UQ_OK, UQ_ERR_DEVICE_FLAG):
        _check(st)
    return int(flags.value)
