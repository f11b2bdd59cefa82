"""The kv-head partition of tensor parallelism, emulated on one GPU.

The pages run the backend at TP = 8 with the KV heads divided between ranks
(flydsl_ultraquant_decode, the end-to-end inter-token-latency comment measured
at TP=8): each rank stores and attends over its own kv heads and their query
heads, and attention needs no exchange between ranks.  Here two "ranks" each
fill their own cache with uq_store from K/V[:, their Hk/2 kv heads] and run
uq_decode on their Hq/2 query heads.  Their caches must equal the matching
head slice of the full cache byte for byte (the store treats every (token,
kv head) alone), and their outputs must match the matching slice of the full
call within the decode tolerance: the split plan sizes its units from the
call's total work, so the two sides may split the sequences differently.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from bit_quantized_kv_gb300 import binding, workloads

from _util import compare, lib, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


@pytest.mark.parametrize("Hq,Hk,ranks", [(32, 4, 2), (64, 4, 2), (48, 8, 4), (64, 8, 8)])
def test_kv_head_slices_reproduce_the_full_call(Hq, Hk, ranks):
    lens = np.array([3000, 17, 640, 1, 1500], np.int32)
    wl = workloads.make_decode_workload("tp", len(lens), Hq, Hk, lens, 200, 16, seed=80 + Hq + ranks)
    dev = "cuda"
    full_cache = torch.zeros((wl.num_blocks, 16, Hk, 272), dtype=torch.uint8, device=dev)
    kv = [workloads.sequence_kv(wl, b, dev) for b in range(wl.B)]
    slots = [torch.from_numpy(workloads.sequence_slots(wl, b)).to(dev) for b in range(wl.B)]
    for b in range(wl.B):
        binding.uq_store(kv[b][0], kv[b][1], full_cache, slots[b])
    q = workloads.query(wl, dev)
    full = run_decode(wl, full_cache, q)
    hk, hq = Hk // ranks, Hq // ranks
    for r in range(ranks):
        heads = slice(r * hk, (r + 1) * hk)
        cache = torch.zeros((wl.num_blocks, 16, hk, 272), dtype=torch.uint8, device=dev)
        for b in range(wl.B):
            binding.uq_store(kv[b][0][:, heads], kv[b][1][:, heads], cache, slots[b])
        assert torch.equal(cache, full_cache[:, :, heads]), f"rank {r}: cache differs from the head slice"
        part = workloads.make_decode_workload("tp_rank", wl.B, hq, hk, lens, 200, 16, seed=0)
        part.block_table = wl.block_table
        part.num_blocks = wl.num_blocks
        q_r = q[:, r * hq:(r + 1) * hq]                   # strided query rows are allowed
        out = run_decode(part, cache, q_r)
        compare(out, full[:, r * hq:(r + 1) * hq].float().cpu().numpy().astype(np.float64))
    assert binding.uq_check_device_error() == 0
