"""Decode at the limits the C ABI accepts, against the fp64 oracle.

A work unit is packed as sequence | split << 16 | kv head << 24, so the
largest batch (B = 65535), the largest split count (S = 256) and the most kv
heads (Hk = 256) each fill one of its fields.  Each case compares output
rows with the oracle's decode of the oracle's own packing of the same
inputs (sampled rows where the batch is large), within the decode tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import bits, compare, fill_cache_gpu, lib, oracle_rows, run_decode

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


def test_largest_batch():
    """65535 sequences of 0 to 5 tokens (8 query heads, one kv head, one
    split): the plan's per-thread chunks, the unit word's sequence field and
    stage 2's row index all reach their largest values."""
    B = 65535
    lens = np.random.default_rng(61).integers(0, 6, size=B).astype(np.int32)
    wl = workloads.make_decode_workload("bigB", B, 8, 1, lens, 1, 1, seed=62)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q)
    assert binding.uq_check_device_error() == 0
    picks = [b for b in range(0, B, 2521)] + [B - 1]
    rows = [(b, r) for b in picks if lens[b] > 0 for r in (0, 7)]
    ref, _ = oracle_rows(wl, q, rows)
    got = torch.stack([out[b, r] for b, r in rows])
    compare(got, ref)
    empty = torch.from_numpy(np.flatnonzero(lens == 0)[:64]).cuda()
    assert torch.count_nonzero(out[empty].float()) == 0


def test_most_splits():
    """One 40000-token sequence with 16 query heads per kv head and S = 256:
    the plan may use every split, so the unit word's split field and stage
    2's merge reach 256 partials."""
    L = 40000
    wl = workloads.make_decode_workload("bigS", 1, 16, 1, np.array([L]), (L + 15) // 16, 256, seed=63)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q)
    assert binding.uq_check_device_error() == 0
    ref, _ = oracle_rows(wl, q, [(0, r) for r in range(16)])
    compare(out[0], ref)


@pytest.mark.parametrize("QG", [6, 16])
def test_most_kv_heads(QG):
    """256 kv heads: the unit word's kv-head field reaches 255."""
    Hk = 256
    lens = np.array([50, 7], np.int32)
    wl = workloads.make_decode_workload("bigH", len(lens), QG * Hk, Hk, lens, 4, 3, seed=64 + QG)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q)
    assert binding.uq_check_device_error() == 0
    rows = [(b, r) for b in range(2) for r in (0, QG - 1, 200 * QG + 3, QG * Hk - 1)]
    ref, _ = oracle_rows(wl, q, rows)
    compare(torch.stack([out[b, r] for b, r in rows]), ref)
