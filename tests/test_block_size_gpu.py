"""Page sizes above 16 tokens (vllm.v1.attention.ops.flydsl_ultraquant_decode,
flydsl_ultraquant_decode_attention: block_size 16..256 accepted).  The
kernels walk rows in 16-token tiles, block_size / 16 of them per page; decode
(with and without a window), multi-query decode and the full-prefix dequant
against the oracle on its own packing of the same inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import bits, compare, fill_cache_gpu, gpu_pages_of_sequence, lib, oracle_cache_for_sequence

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("bs", [32, 64, 256])
@pytest.mark.parametrize("Hq,Hk,window", [(8, 1, 0), (12, 2, 50), (32, 2, 0)])
def test_decode_matches_oracle(bs, Hq, Hk, window):
    lens = np.array([1, 15, 16, 33, 100, 257, 700, 1111, 0, 513], np.int32)
    maxb = -(-1111 // bs) + 1
    S = 8
    wl = workloads.make_decode_workload("bs", len(lens), Hq, Hk, lens, maxb, S, seed=bs + Hq,
                                        spare_blocks=2, block_size=bs)
    cache = fill_cache_gpu(wl)
    ref_cache = _oracle_cache(wl)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    q = workloads.query(wl, "cuda")
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, Hq, 256, S), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.B, Hq, 256), dtype=torch.bfloat16, device="cuda")
    binding.uq_decode_ex(q, cache, bt, sl, wl.scale, None, window, S, ws, out)
    assert binding.uq_check_device_error() == 0
    ref = oracle.decode(bits(q), ref_cache, wl.block_table, wl.seq_lens, wl.scale, window=window)
    compare(out, ref)


@pytest.mark.parametrize("bs", [32, 128])
def test_multi_query_matches_oracle(bs):
    cached, q_len, S = 600, 4, 8
    L = cached + q_len
    P = -(-L // bs)
    wl = workloads.make_decode_workload("bsmq", 1, 16, 2, np.array([L]), P + 1, S, seed=bs,
                                        block_size=bs)
    cache = fill_cache_gpu(wl)
    ref_cache = oracle_cache_for_sequence(wl, 0)
    assert np.array_equal(gpu_pages_of_sequence(cache, wl, 0), ref_cache)
    q = workloads.chunk_query(wl, q_len, "cuda")
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(q_len, wl.Hq, 256, S), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out)
    table = np.tile(np.arange(P, dtype=np.int32), (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    compare(out, oracle.decode(bits(q), ref_cache, table, lens, wl.scale))


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_full_dequant_bit_exact(bs):
    rng = np.random.default_rng(bs)
    nb, Hk = 7, 3
    cache = rng.integers(0, 256, size=(nb, bs, Hk, 272), dtype=np.uint8)
    table = np.array([5, 0, 6, 2], np.int32)
    n = len(table)
    k = torch.empty((Hk, n * bs, 256), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    binding.uq_full_dequant(torch.from_numpy(cache).cuda(), torch.from_numpy(table).cuda(), k, v)
    assert binding.uq_check_device_error() == 0
    kr, vr, bad = oracle.full_dequant(cache, table)
    assert bad == 0
    assert np.array_equal(bits(k), kr) and np.array_equal(bits(v), vr)
