"""uq_decode_static_scratch: decode for callers that cannot allocate.

Some integrations cannot give uq_decode a workspace (a plugin whose enqueue
step must not call cudaMalloc, a host that keeps every byte of device memory
in its own pool).  For them the library offers uq_decode_static_scratch,
which keeps the split partials in a fixed 32 MiB array owned by the library.
This test calls it through the C ABI and checks that it returns what
uq_decode returns, within the decode tolerance used by the other tests, on
two calls in a row (the second call finds the first call's partials still in
the shared array), and that an oversize batch is refused.  The file is named
so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from bit_quantized_kv_gb300 import binding, workloads

from _util import compare, fill_cache_gpu, lib, run_decode

pytestmark = pytest.mark.gpu


def _static_scratch_call(wl, cache, q, splits, seq_lens=None):
    """Call the C entry point directly through ctypes (no workspace argument)."""
    L = lib()
    dev = cache.device
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens if seq_lens is None else seq_lens).to(dev)
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream or None
    st = L.uq_decode_static_scratch(q.data_ptr(), cache.data_ptr(), bt.data_ptr(), sl.data_ptr(),
                                    ctypes.c_float(wl.scale), splits, out.data_ptr(), wl.B, wl.Hq,
                                    wl.Hk, wl.D, wl.num_blocks, wl.block_size, wl.max_blocks, 272,
                                    q.stride(0), q.stride(1), stream)
    assert st == binding.UQ_OK, binding.uq_last_error()
    torch.cuda.synchronize()
    return out


def _reference(got, expect):
    compare(got, expect.float().cpu().numpy().astype(np.float64))


def test_static_scratch_matches_uq_decode_two_calls_in_a_row():
    lib()
    lens = np.array([1, 17, 300, 1500, 4000, 33, 0, 777], np.int32)
    wl = workloads.make_decode_workload("noalloc", len(lens), 48, 8, lens, 256, 16, seed=61)
    cache = fill_cache_gpu(wl)
    q1 = workloads.query(wl, "cuda", step=0)
    q2 = workloads.query(wl, "cuda", step=1)
    # first call, then a second call with other queries and shorter lengths
    got1 = _static_scratch_call(wl, cache, q1, wl.splits)
    _reference(got1, run_decode(wl, cache, q1))
    short = np.minimum(lens, 500).astype(np.int32)
    got2 = _static_scratch_call(wl, cache, q2, wl.splits, seq_lens=short)
    _reference(got2, run_decode(wl, cache, q2, seq_lens=short))
    assert binding.uq_check_device_error() == 0


def test_static_scratch_at_its_size_limit():
    # B * Hq * S = 32 * 32 * 31 = 31744 rows fit the 32 MiB array
    wl = workloads.decode_workload("batch")
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    for _ in range(2):
        _reference(_static_scratch_call(wl, cache, q, 31), run_decode(wl, cache, q, splits=31))


def test_static_scratch_rejects_oversize_batch():
    wl = workloads.decode_workload("batch")              # 32 * 32 * 32 = 32768 rows do not
    L = lib()
    cache = torch.zeros((1, 16, wl.Hk, 272), dtype=torch.uint8, device="cuda")
    q = torch.zeros((wl.B, wl.Hq, 256), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    bt = torch.zeros((wl.B, 1), dtype=torch.int32, device="cuda")
    sl = torch.zeros((wl.B,), dtype=torch.int32, device="cuda")
    st = L.uq_decode_static_scratch(q.data_ptr(), cache.data_ptr(), bt.data_ptr(), sl.data_ptr(),
                                    ctypes.c_float(0.0625), 32, out.data_ptr(), wl.B, wl.Hq, wl.Hk,
                                    256, 1, 16, 1, 272, q.stride(0), q.stride(1), None)
    assert st == binding.UQ_ERR_WORKSPACE_TOO_SMALL
    assert "32 MiB" in binding.uq_last_error()
