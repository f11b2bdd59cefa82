"""GPU parity of uq_decode_ex (attention sinks and a sliding window, the
sinks / sliding_window of vllm.v1.attention.backends.ultraquant_attn,
UltraQuantAttentionImpl) and of uq_decode_multi_query with both, against the
fp64 oracle on its own packing of the same inputs."""
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


def _decode_ex(wl, cache, q, sinks, window, S):
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, 256, S), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.B, wl.Hq, 256), dtype=torch.bfloat16, device="cuda")
    sk = None if sinks is None else torch.from_numpy(sinks.astype(np.float32)).cuda()
    binding.uq_decode_ex(q, cache, bt, sl, wl.scale, sk, window, S, ws, out)
    return out


@pytest.mark.parametrize("Hq,Hk", [(8, 1), (12, 2), (32, 2)])
@pytest.mark.parametrize("window,with_sinks", [(1, False), (16, True), (17, False), (100, True),
                                                (5000, True), (0, True)])
def test_window_and_sinks_match_oracle(Hq, Hk, window, with_sinks):
    lens = np.array([1, 15, 16, 17, 100, 257, 700, 1111, 0, 33], np.int32)
    S = 8
    wl = workloads.make_decode_workload("ws", len(lens), Hq, Hk, lens, 80, S, seed=90 + Hq + window,
                                        spare_blocks=3)
    cache = fill_cache_gpu(wl)
    ref_cache = _oracle_cache(wl)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    q = workloads.query(wl, "cuda")
    sinks = np.random.default_rng(window + Hq).standard_normal(Hq) * 2.0 if with_sinks else None
    out = _decode_ex(wl, cache, q, sinks, window, S)
    assert binding.uq_check_device_error() == 0
    ref = oracle.decode(bits(q), ref_cache, wl.block_table, wl.seq_lens, wl.scale,
                        sinks=sinks, window=window)
    compare(out, ref)


def test_no_sinks_no_window_equals_uq_decode():
    wl = workloads.decode_workload("tiny")
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    got = _decode_ex(wl, cache, q, None, 0, wl.splits)
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, 256, wl.splits), dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(got)
    binding.uq_decode(q, cache, bt, sl, wl.scale, wl.splits, ws, ref)
    assert torch.equal(got, ref)


def test_window_longer_than_every_sequence_changes_nothing():
    lens = np.array([40, 900, 3000], np.int32)
    wl = workloads.make_decode_workload("ws", 3, 16, 2, lens, 200, 8, seed=95)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    assert torch.equal(_decode_ex(wl, cache, q, None, 3000, 8), _decode_ex(wl, cache, q, None, 0, 8))


def test_multi_query_with_window_and_sinks():
    cached, q_len, S, window = 300, 5, 8, 37
    L = cached + q_len
    P = (L + 15) // 16
    wl = workloads.make_decode_workload("mqws", 1, 16, 2, np.array([L]), P + 1, S, seed=96)
    cache = fill_cache_gpu(wl)
    ref_cache = oracle_cache_for_sequence(wl, 0)
    assert np.array_equal(gpu_pages_of_sequence(cache, wl, 0), ref_cache)
    q = workloads.chunk_query(wl, q_len, "cuda")
    sinks = np.random.default_rng(3).standard_normal(wl.Hq) * 2.0
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(q_len, wl.Hq, 256, S), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out,
                                  sinks=torch.from_numpy(sinks.astype(np.float32)).cuda(),
                                  sliding_window=window)
    assert binding.uq_check_device_error() == 0
    table = np.tile(np.arange(P, dtype=np.int32), (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    ref = oracle.decode(bits(q), ref_cache, table, lens, wl.scale, sinks=sinks, window=window)
    compare(out, ref)
