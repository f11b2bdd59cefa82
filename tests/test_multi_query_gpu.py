"""GPU parity of uq_decode_multi_query, the continuation-chunk attention of
vllm.v1.attention.backends.ultraquant_attn, UltraQuantAttentionImpl.
_prefill_attention (chunks up to _CONTINUATION_DECODE_THRESHOLD: the decode
kernel over synthetic seq_lens = arange(cached + 1, seq_len + 1) and an
expanded block table).  Reference: the fp64 oracle's decode over exactly that
synthetic batch, built from the oracle's own packing of the same inputs."""
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


def _mq(wl, cache, q, cached, S):
    q_len = q.shape[0]
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(max(q_len, 1), wl.Hq, 256, S), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(q)
    binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out)
    return out


@pytest.mark.parametrize("cached,q_len,Hq,Hk,S", [
    (0, 1, 8, 1, 4),          # the first token of a sequence
    (15, 2, 48, 8, 1),        # chunk starts at the end of a page
    (16, 3, 12, 2, 8),        # chunk starts on a page boundary, GQA 6
    (17, 8, 32, 2, 32),       # GQA 16
    (777, 5, 8, 1, 3),
    (5000, 4, 64, 8, 32),
])
def test_matches_oracle_synthetic_batch(cached, q_len, Hq, Hk, S):
    L = cached + q_len
    P = (L + 15) // 16
    wl = workloads.make_decode_workload("mq", 1, Hq, Hk, np.array([L]), P + 2, S,
                                        seed=60 + cached % 97 + q_len, spare_blocks=3)
    cache = fill_cache_gpu(wl)
    q = workloads.chunk_query(wl, q_len, "cuda")
    out = _mq(wl, cache, q, cached, S)
    assert binding.uq_check_device_error() == 0
    ref_cache = oracle_cache_for_sequence(wl, 0)
    assert np.array_equal(gpu_pages_of_sequence(cache, wl, 0), ref_cache)
    table = np.tile(np.arange(P, dtype=np.int32), (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    ref = oracle.decode(bits(q), ref_cache, table, lens, wl.scale)
    compare(out, ref)


def _agree(a: torch.Tensor, b: torch.Tensor):
    """Two GPU results of the same attention within the decode tolerance
    (max-abs 1e-2, relative L2 5e-3).  The multi-query entry packs two chunk
    positions into one 16-row unit (6 or 8 query heads per kv head), so it
    runs other tiles and splits than uq_decode and is not bit-identical."""
    compare(a, b.detach().float().cpu().numpy().astype(np.float64).reshape(a.shape))


def test_equals_decode_on_the_expanded_batch():
    """Agrees with uq_decode given the materialised synthetic batch."""
    cached, q_len, S = 2047, 6, 16
    wl = workloads.make_decode_workload("mq", 1, 48, 8, np.array([cached + q_len]), 140, S, seed=71)
    cache = fill_cache_gpu(wl)
    q = workloads.chunk_query(wl, q_len, "cuda")
    out = _mq(wl, cache, q, cached, S)
    bt = torch.from_numpy(np.tile(wl.block_table[0], (q_len, 1))).cuda()
    sl = torch.arange(cached + 1, cached + q_len + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.uq_decode_workspace_bytes(q_len, wl.Hq, 256, S), dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(q)
    binding.uq_decode(q, cache, bt, sl, wl.scale, S, ws, ref)
    _agree(out, ref)


def test_last_row_equals_plain_decode():
    """Row q_len - 1 sees the whole sequence: the same as decoding that query alone."""
    cached, q_len, S = 900, 3, 8
    wl = workloads.make_decode_workload("mq", 1, 16, 2, np.array([cached + q_len]), 60, S, seed=72)
    cache = fill_cache_gpu(wl)
    q = workloads.chunk_query(wl, q_len, "cuda")
    out = _mq(wl, cache, q, cached, S)
    bt = torch.from_numpy(wl.block_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(1, wl.Hq, 256, S), dtype=torch.uint8, device="cuda")
    ref = torch.empty((1, wl.Hq, 256), dtype=torch.bfloat16, device="cuda")
    binding.uq_decode(q[q_len - 1:].contiguous(), cache, bt, sl, wl.scale, S, ws, ref)
    _agree(out[q_len - 1], ref[0])


def test_full_size_sampled_rows():
    """The benchmark's chunk (131072 cached + 8 tokens, GQA 8): every chunk
    row, the first and last query head of each kv head group sampled."""
    wl, cached, q_len = workloads.multi_query_workload("mq")
    cache = fill_cache_gpu(wl)
    q = workloads.chunk_query(wl, q_len, "cuda")
    out = _mq(wl, cache, q, cached, wl.splits)
    assert binding.uq_check_device_error() == 0
    ref_cache = oracle_cache_for_sequence(wl, 0)
    P = ref_cache.shape[0]
    heads = [0, 7, 31, 63]
    rows = np.array([[i, r] for i in range(q_len) for r in heads], np.int32)
    table = np.tile(np.arange(P, dtype=np.int32), (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    ref = oracle.decode(bits(q), ref_cache, table, lens, wl.scale, rows=rows)
    got = torch.stack([out[i, r] for i, r in rows])
    compare(got, ref)


def test_empty_chunk_is_a_noop():
    wl = workloads.make_decode_workload("mq", 1, 8, 1, np.array([16]), 2, 4, seed=73)
    cache = torch.zeros((wl.num_blocks, 16, 1, 272), dtype=torch.uint8, device="cuda")
    q = torch.empty((0, 8, 256), dtype=torch.bfloat16, device="cuda")
    _mq(wl, cache, q, 16, 4)
    assert binding.uq_check_device_error() == 0


@pytest.mark.parametrize("seed", range(24))
def test_random_chunks_match_oracle(seed):
    """Seeded random chunks: 6, 8 or 16 query heads per kv head, 1 to 3 kv
    heads, 0 to 2999 cached tokens, 1 to 8 chunk rows, 1 to 32 splits, and
    sometimes a sliding window.  Covers both multi-query kernels (packed
    chunk rows without a window, and the general one with it) against the
    oracle's decode of the synthetic batch."""
    rng = np.random.default_rng(7000 + seed)
    QG = int(rng.choice([6, 8, 16]))
    Hk = int(rng.integers(1, 4))
    cached = int(rng.integers(0, 3000))
    q_len = int(rng.integers(1, 9))
    S = int(rng.integers(1, 33))
    window = int(rng.choice([0, 0, 50, 700]))
    L = cached + q_len
    P = (L + 15) // 16
    wl = workloads.make_decode_workload("mq", 1, QG * Hk, Hk, np.array([L]), P + 2, S, seed=300 + seed,
                                        spare_blocks=3)
    cache = fill_cache_gpu(wl)
    q = workloads.chunk_query(wl, q_len, "cuda")
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(q_len, wl.Hq, 256, S), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out, sliding_window=window)
    assert binding.uq_check_device_error() == 0
    ref_cache = oracle_cache_for_sequence(wl, 0)
    table = np.tile(np.arange(P, dtype=np.int32), (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    compare(out, oracle.decode(bits(q), ref_cache, table, lens, wl.scale, window=window))
