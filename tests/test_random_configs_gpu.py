"""Seeded random decode configurations against the fp64 oracle.

Each case draws its own shape: 6, 8 or 16 query heads per kv head, 1 to 3
kv heads, 1 to 8 sequences of 0 to 699 tokens (some empty), 16-, 32- or
64-token pages, 1 to 16 splits, and sometimes a sliding window and sink
logits.  The cache is filled with uq_store, checked byte for byte against
the oracle's own packing, and uq_decode_ex is compared element by element
with the oracle's fp64 attention over that cache, within the decode
tolerance.  A second test runs far K blocks (scales 2^40 above the rest of
their token) through uq_decode_static_scratch, so that the exact pass also
runs with the library's own scratch.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import bits, compare, fill_cache_gpu, lib

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


def _oracle_cache(wl):
    ref = np.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), np.uint8)
    for b in range(wl.B):
        if wl.seq_lens[b] == 0:
            continue
        k, v = workloads.sequence_kv(wl, b, "cuda")
        oracle.store(bits(k), bits(v), workloads.sequence_slots(wl, b), ref)
    return ref


@pytest.mark.parametrize("seed", range(64))
def test_random_configuration_matches_oracle(seed):
    rng = np.random.default_rng(4000 + seed)
    QG = int(rng.choice([6, 8, 16]))
    Hk = int(rng.integers(1, 4))
    Hq = QG * Hk
    B = int(rng.integers(1, 9))
    lens = rng.integers(0, 700, size=B).astype(np.int32)
    lens[rng.random(B) < 0.15] = 0
    block_size = int(rng.choice([16, 32, 64]))
    S = int(rng.integers(1, 17))
    window = int(rng.choice([0, 0, 1, 37, 300]))
    sinks = rng.standard_normal(Hq) * 3.0 if rng.random() < 0.4 else None
    max_blocks = max(1, int((int(lens.max()) + block_size - 1) // block_size)) + int(rng.integers(0, 3))
    wl = workloads.make_decode_workload("rand", B, Hq, Hk, lens, max_blocks, S, seed=500 + seed,
                                        spare_blocks=2, block_size=block_size)
    cache = fill_cache_gpu(wl)
    ref_cache = _oracle_cache(wl)
    assert np.array_equal(cache.cpu().numpy(), ref_cache), "packed cache differs from the oracle's"
    q = workloads.query(wl, "cuda")
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(B, Hq, D, S), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    sk = None if sinks is None else torch.from_numpy(sinks.astype(np.float32)).cuda()
    binding.uq_decode_ex(q, cache, bt, sl, wl.scale, sk, window, S, ws, out)
    assert binding.uq_check_device_error() == 0
    ref = oracle.decode(bits(q), ref_cache, wl.block_table, wl.seq_lens, wl.scale, sinks=sinks,
                        window=window)
    compare(out, ref)


@pytest.mark.parametrize("Hq,Hk", [(8, 1), (12, 2), (32, 2)])
def test_far_k_blocks_through_the_static_scratch(Hq, Hk):
    """K blocks 2^40 above the rest of their token on every token, with
    query rows zero there: the split-KV kernel lists every unit for the
    exact pass, whose redo list lives in the library's static scratch."""
    rng = np.random.default_rng(4100 + Hq)
    lens = np.array([5, 333, 90, 700], np.int32)
    max_blocks = int((lens.max() + 15) // 16)
    wl = workloads.make_decode_workload("far", len(lens), Hq, Hk, lens, max_blocks, 6, seed=41,
                                        spare_blocks=2)
    n = int(lens.sum())
    kr = rng.standard_normal((n, Hk, D)).astype(np.float32)
    kr[:, :, 160:192] *= np.float32(2.0 ** 40)
    vv = rng.standard_normal((n, Hk, D)).astype(np.float32)
    slots = np.concatenate([workloads.sequence_slots(wl, b) for b in range(wl.B)])
    cache = torch.zeros((wl.num_blocks, 16, Hk, 272), dtype=torch.uint8, device="cuda")
    binding.uq_store_rotated_f32(torch.from_numpy(kr).cuda(), torch.from_numpy(vv).cuda(), cache,
                                 torch.from_numpy(slots).cuda())
    ref_cache = np.zeros((wl.num_blocks, 16, Hk, 272), np.uint8)
    oracle.store_f32(kr, vv, slots, ref_cache)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    qp[..., 160:192] = 0.0
    q_bits = oracle.bf16_round_array(qp @ oracle.hadamard(D))
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    out = torch.empty((wl.B, Hq, D), dtype=torch.bfloat16, device="cuda")
    binding.uq_decode_static_scratch(q, cache, bt, sl, wl.scale, wl.splits, out)
    assert binding.uq_check_device_error() == 0
    compare(out, oracle.decode(q_bits, ref_cache, wl.block_table, wl.seq_lens, wl.scale))
