"""The decode kernel's bounded waits give up instead of hanging.

Stage 1 waits for each page copy on an mbarrier with a capped number of
try_wait attempts; when the cap runs out the warp records UQ_DEVERR_TIMEOUT in
the device error word, waits (again bounded) for its copies still in flight,
and the CTA stops taking work units, so the call returns and the context stays
usable.  The flydsl_ultraquant_decode page guards its buffers with host-side
warnings only (_SegmBufPool's growth warning during graph capture); here the
device-side give-up path is exercised directly.

A test-only variant of the library (built beside libuq.so as
libuq_stuck_tile.so, never loaded by the package) announces the first page of
work unit 0 to its barrier without copying it, and shortens the waits to a
fraction of a millisecond.  No copy is ever in flight for that stage, so the
GPU only sees a barrier phase that does not complete.  The test runs the
variant on the 8-row kernel (6 and 8 query heads per kv head) and on the
16-row kernel, whose O^T lives in tensor memory and whose warps must give up
together so that their warp-collective tensor-memory instructions stay
converged.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from bit_quantized_kv_gb300 import binding, workloads
from bit_quantized_kv_gb300.build import build

from _util import compare, fill_cache_gpu, lib, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def stuck():
    lib()
    return binding.load(build(variant="stuck_tile"))


def _variant_decode(L, wl, cache, q):
    dev = cache.device
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, 256, wl.splits), dtype=torch.uint8, device=dev)
    out = torch.full((wl.B, wl.Hq, 256), float("nan"), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream or None
    st = L.uq_decode(q.data_ptr(), cache.data_ptr(), bt.data_ptr(), sl.data_ptr(), ctypes.c_float(wl.scale),
                     wl.splits, ws.data_ptr(), ws.numel(), out.data_ptr(), wl.B, wl.Hq, wl.Hk, 256,
                     wl.num_blocks, wl.block_size, wl.max_blocks, 272, q.stride(0), q.stride(1), stream)
    assert st == binding.UQ_OK, L.uq_last_error().decode()
    flags = ctypes.c_uint(0)
    st = L.uq_check_device_error(stream, ctypes.byref(flags))
    assert st in (binding.UQ_OK, binding.UQ_ERR_DEVICE_FLAG)
    return out, int(flags.value)


@pytest.mark.parametrize("Hq,Hk", [(8, 1), (12, 2), (32, 2)])
def test_a_wait_that_runs_out_is_reported_and_the_call_returns(stuck, Hq, Hk):
    lens = np.array([900, 64, 300, 17, 2000, 5], np.int32)
    wl = workloads.make_decode_workload("stuck", len(lens), Hq, Hk, lens, 125, 4, seed=70 + Hq)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out, flags = _variant_decode(stuck, wl, cache, q)
    assert flags & binding.UQ_DEVERR_TIMEOUT, f"flags {flags:#x}"
    assert torch.isfinite(out.float()).all()
    # Work unit 0 is the longest sequence's first split of kv head 0: only
    # its query heads lose the pages of the warp that gave up.  Every other
    # row, including those of units that the stopped CTA would have taken
    # next, matches the product library.
    good = run_decode(wl, cache, q)
    assert binding.uq_check_device_error() == 0      # the context is still usable
    b0 = int(np.argmax(lens))
    keep = np.ones((wl.B, wl.Hq), bool)
    keep[b0, :Hq // Hk] = False
    keep_t = torch.from_numpy(keep).cuda()
    compare(out[keep_t], good[keep_t].float().cpu().numpy().astype(np.float64))
    # a second call of the variant gives up the same way, and clears nothing else
    out2, flags2 = _variant_decode(stuck, wl, cache, q)
    assert flags2 & binding.UQ_DEVERR_TIMEOUT
    compare(out2[keep_t], good[keep_t].float().cpu().numpy().astype(np.float64))
