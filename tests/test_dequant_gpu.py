"""GPU parity of uq_full_dequant (the prefix buffers of the continuation
prefill, vllm.v1.attention.backends.ultraquant_attn,
UltraQuantAttentionImpl._ultraquant_continuation_prefill) against the fp64
CPU oracle: bit-exact bf16, on arbitrary cache bytes and on caches written
by uq_store."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import fill_cache_gpu, gpu_pages_of_sequence, lib, oracle_cache_for_sequence

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


def _run(cache_gpu: torch.Tensor, table: np.ndarray):
    Hk = cache_gpu.shape[2]
    n = len(table)
    bt = torch.from_numpy(np.ascontiguousarray(table, np.int32)).cuda()
    k = torch.full((Hk, n * 16, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    v = torch.full_like(k, float("nan"))
    binding.uq_full_dequant(cache_gpu, bt, k, v)
    return k, v


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("nb,Hk,table", [
    (4, 1, [2]),
    (9, 3, [4, 0, 8, 2, 7]),
    (40, 8, list(np.random.default_rng(3).permutation(40)[:37])),
])
def test_random_bytes_bit_exact(nb, Hk, table):
    """Every code and every scale byte, 0 and 254..255 included."""
    rng = np.random.default_rng(nb * 100 + Hk)
    cache = rng.integers(0, 256, size=(nb, 16, Hk, 272), dtype=np.uint8)
    table = np.array(table, np.int32)
    k, v = _run(torch.from_numpy(cache).cuda(), table)
    assert binding.uq_check_device_error() == 0
    kr, vr, bad = oracle.full_dequant(cache, table)
    assert bad == 0
    assert np.array_equal(_bits(k), kr) and np.array_equal(_bits(v), vr)


def test_stored_cache_bit_exact():
    """A cache written by uq_store; the oracle dequantises its own packing of
    the same bf16 inputs (checked byte for byte against the GPU's pages)."""
    wl = workloads.dequant_workload("dequant_small")
    cache = fill_cache_gpu(wl)
    ref_cache = oracle_cache_for_sequence(wl, 0)                 # page i at cache page i
    assert np.array_equal(gpu_pages_of_sequence(cache, wl, 0), ref_cache)
    n = ref_cache.shape[0]
    k, v = _run(cache, wl.block_table[0, :n])
    kr, vr, bad = oracle.full_dequant(ref_cache, np.arange(n, dtype=np.int32))
    assert bad == 0
    assert np.array_equal(_bits(k), kr) and np.array_equal(_bits(v), vr)


def test_bad_page_is_zeroed_and_flagged():
    rng = np.random.default_rng(5)
    cache = rng.integers(0, 256, size=(6, 16, 2, 272), dtype=np.uint8)
    table = np.array([1, 99, 4, -3], np.int32)
    k, v = _run(torch.from_numpy(cache).cuda(), table)
    assert binding.uq_check_device_error() & binding.UQ_DEVERR_BAD_PAGE
    kr, vr, bad = oracle.full_dequant(cache, table)
    assert bad == 2
    assert np.array_equal(_bits(k), kr) and np.array_equal(_bits(v), vr)


def test_zero_pages_is_a_noop():
    cache = torch.zeros((2, 16, 1, 272), dtype=torch.uint8, device="cuda")
    k = torch.empty((1, 0, 256), dtype=torch.bfloat16, device="cuda")
    binding.uq_full_dequant(cache, torch.zeros(0, dtype=torch.int32, device="cuda"), k, k.clone())
    assert binding.uq_check_device_error() == 0


def test_full_size_sampled_pages():
    """The benchmark's workload (32768 tokens, 8 kv heads) in the launch the
    benchmark times; 24 sampled pages compared bit for bit against the
    oracle's dequantisation of its own packing."""
    wl = workloads.dequant_workload("dequant")
    cache = fill_cache_gpu(wl)
    table = wl.block_table[0]
    k, v = _run(cache, table)
    assert binding.uq_check_device_error() == 0
    ref_cache = oracle_cache_for_sequence(wl, 0)
    pages = np.sort(np.random.default_rng(9).choice(len(table), 24, replace=False))
    gpu_pages = cache.index_select(0, torch.as_tensor(table[pages].astype(np.int64), device="cuda"))
    assert np.array_equal(gpu_pages.cpu().numpy(), ref_cache[pages])
    kr, vr, _ = oracle.full_dequant(ref_cache, pages.astype(np.int32))
    kb, vb = _bits(k), _bits(v)
    for i, p in enumerate(pages):
        assert np.array_equal(kb[:, 16 * p:16 * p + 16], kr[:, 16 * i:16 * i + 16])
        assert np.array_equal(vb[:, 16 * p:16 * p + 16], vr[:, 16 * i:16 * i + 16])
