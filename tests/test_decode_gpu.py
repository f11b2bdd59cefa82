"""GPU parity of uq_decode against the fp64 CPU oracle (max-abs 1e-2,
relative L2 5e-3 on the bf16 output), on the oracle's own packed cache:
every cache page the GPU reads is first checked byte for byte against the
oracle's packing of the same seeded inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import (bits, compare, fill_cache_gpu, gpu_pages_of_sequence, lib,
                   oracle_cache_for_sequence, run_decode)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


def _full_parity(wl, splits=None):
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q, splits=splits)
    assert binding.uq_check_device_error() == 0
    # the oracle's own cache, laid out with the same page table
    ref_cache = np.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), np.uint8)
    for b in range(wl.B):
        if wl.seq_lens[b] == 0:
            continue
        k, v = workloads.sequence_kv(wl, b, "cuda")
        oracle.store(bits(k), bits(v), workloads.sequence_slots(wl, b), ref_cache)
    assert np.array_equal(cache.cpu().numpy(), ref_cache), "packed cache differs from the oracle"
    ref = oracle.decode(bits(q), ref_cache, wl.block_table, wl.seq_lens, wl.scale)
    return compare(out, ref)


def test_tiny_full_parity():
    _full_parity(workloads.decode_workload("tiny"))


@pytest.mark.parametrize("Hq,Hk", [(8, 1), (12, 2), (32, 2)])   # GQA 8, 6, 16
@pytest.mark.parametrize("splits", [1, 3, 32])
def test_ragged_lengths_all_group_sizes(Hq, Hk, splits):
    lens = np.array([1, 15, 16, 17, 100, 257, 700, 1111, 0, 33], np.int32)
    wl = workloads.make_decode_workload("ragged", len(lens), Hq, Hk, lens, 80, splits,
                                        seed=20 + Hq + splits, spare_blocks=3)
    _full_parity(wl)


def test_single_token_sequences():
    lens = np.ones(7, np.int32)
    wl = workloads.make_decode_workload("ones", 7, 16, 1, lens, 1, 4, seed=31)
    _full_parity(wl)


def test_larger_scale_sharper_softmax():
    lens = np.array([300, 2000], np.int32)
    wl = workloads.make_decode_workload("sharp", 2, 8, 1, lens, 125, 8, seed=32, scale=0.25)
    _full_parity(wl)


def test_batch_workload_parity():
    """B=32, Hq=32, Hk=4, L in [1024, 8192], S=32: every output row."""
    _full_parity(workloads.decode_workload("batch"))


def _sampled_parity(name, n_rows=24):
    wl = workloads.decode_workload(name)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q)
    assert binding.uq_check_device_error() == 0
    rng = np.random.default_rng(5)
    order = np.argsort(wl.seq_lens)
    seqs = sorted(set([int(order[0]), int(order[-1]), int(order[len(order) // 2])] +
                      list(rng.choice(wl.B, 3, replace=False))))
    qb = bits(q)
    got_rows, ref_rows = [], []
    for b in seqs:
        ref_cache = oracle_cache_for_sequence(wl, b)
        assert np.array_equal(gpu_pages_of_sequence(cache, wl, b), ref_cache), f"seq {b} bytes differ"
        heads = sorted(set([0, wl.Hq - 1] + list(rng.choice(wl.Hq, max(1, n_rows // len(seqs) - 2),
                                                            replace=False))))
        rows = np.array([[0, r] for r in heads], np.int32)
        P = ref_cache.shape[0]
        ref = oracle.decode(qb[b:b + 1], ref_cache, np.arange(P, dtype=np.int32)[None],
                            wl.seq_lens[b:b + 1], wl.scale, rows=rows)
        ref_rows.append(ref)
        got_rows.append(out[b, heads])
    compare(torch.cat(got_rows), np.concatenate(ref_rows))


def test_outlier_long_sampled_parity():
    _sampled_parity("outlier_long")


def test_skewed_sampled_parity():
    _sampled_parity("skewed")


def test_cuda_graph_replay_with_new_lengths():
    """Capture once, replay with different seq_lens / block_table contents."""
    wl = workloads.make_decode_workload("graph", 6, 64, 4, np.array([40, 900, 3000, 17, 2048, 555]),
                                        200, 8, seed=41)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    dev = "cuda"
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, 256, wl.splits), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.B, wl.Hq, 256), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        binding.uq_decode(q, cache, bt, sl, wl.scale, wl.splits, ws, out)   # warm-up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        binding.uq_decode(q, cache, bt, sl, wl.scale, wl.splits, ws, out)
    for new_lens in ([40, 900, 3000, 17, 2048, 555], [1, 2, 3000, 0, 100, 555], [16, 32, 48, 64, 80, 96]):
        nl = np.array(new_lens, np.int32)
        sl.copy_(torch.from_numpy(nl))
        graph.replay()
        torch.cuda.synchronize()
        eager = run_decode(wl, cache, q, seq_lens=nl)
        assert torch.equal(out, eager)
    assert binding.uq_check_device_error() == 0


@pytest.mark.parametrize("Hq", [8, 16])
def test_bad_page_id_is_flagged_and_skipped(Hq):
    wl = workloads.make_decode_workload("bad", 2, Hq, 1, np.array([64, 64]), 4, 2, seed=43)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    bt = wl.block_table.copy()
    bt[1, 2] = wl.num_blocks + 100         # out of range: that page's tokens are skipped
    out = run_decode(wl, cache, q, block_table=bt)
    flags = binding.uq_check_device_error()
    assert flags & binding.UQ_DEVERR_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    # sequence 0 is unaffected
    ref = run_decode(wl, cache, q)
    assert torch.equal(out[0], ref[0])


def test_length_beyond_table_is_clamped():
    wl = workloads.make_decode_workload("clamp", 1, 8, 1, np.array([64]), 4, 2, seed=44)
    cache = fill_cache_gpu(wl)
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q, seq_lens=np.array([10_000], np.int32))
    ref = run_decode(wl, cache, q)
    assert torch.equal(out, ref)


def test_empty_batch_and_zero_lengths():
    wl = workloads.make_decode_workload("zeros", 3, 16, 2, np.array([0, 0, 0]), 2, 4, seed=45)
    cache = torch.zeros((1, 16, 2, 272), dtype=torch.uint8, device="cuda")
    q = workloads.query(wl, "cuda")
    out = run_decode(wl, cache, q)
    assert not out.float().abs().sum().item()
