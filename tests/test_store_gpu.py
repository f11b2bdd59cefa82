"""GPU parity of the store kernel against the CPU oracle: packed cache bytes
must be bit-exact, both end to end (bf16 K rotated on the GPU) and for the
quantise-and-pack step alone (pre-rotated fp32 K)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import bits, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


def _oracle_store(k, v, slots, shape):
    cache = np.zeros(shape, np.uint8)
    oracle.store(bits(k), bits(v), slots.cpu().numpy(), cache)
    return cache


def test_store_small_bit_exact():
    wl = workloads.store_workload("store_small")
    k, v, slots = workloads.store_inputs(wl, "cuda")
    shape = (wl.num_blocks, wl.block_size, wl.Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store(k, v, cache, slots)
    assert binding.uq_check_device_error() == 0
    assert np.array_equal(cache.cpu().numpy(), _oracle_store(k, v, slots, shape))


@pytest.mark.parametrize("N,Hk", [(1, 1), (3, 2), (33, 5), (257, 8)])
def test_store_ragged_row_counts(N, Hk):
    g = torch.Generator(device="cuda").manual_seed(100 + N)
    k = torch.randn((N, Hk, 256), generator=g, device="cuda").to(torch.bfloat16)
    v = (torch.randn((N, Hk, 256), generator=g, device="cuda") * 3).to(torch.bfloat16)
    nb = (N + 15) // 16 + 1
    slots = torch.randperm(nb * 16, generator=g, device="cuda")[:N].to(torch.int64)
    shape = (nb, 16, Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store(k, v, cache, slots)
    assert np.array_equal(cache.cpu().numpy(), _oracle_store(k, v, slots, shape))


@pytest.mark.parametrize("N,Hk", [(9000, 5), (5000, 7)])
def test_store_several_passes_of_the_persistent_grid(N, Hk):
    """More (token, kv head) rows than the resident CTAs take in one pass
    (3 per SM x 32 rows), with Hk not dividing the pass, so each group's
    token and head advance with a carry; some slots negative, one out of
    range."""
    g = torch.Generator(device="cuda").manual_seed(200 + Hk)
    k = torch.randn((N, Hk, 256), generator=g, device="cuda").to(torch.bfloat16)
    v = (torch.randn((N, Hk, 256), generator=g, device="cuda") * 2).to(torch.bfloat16)
    nb = (N + 15) // 16 + 3
    slots = torch.randperm(nb * 16, generator=g, device="cuda")[:N].to(torch.int64)
    slots[::97] = -1
    slots[N // 2] = nb * 16 + 5
    shape = (nb, 16, Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store(k, v, cache, slots)
    assert binding.uq_check_device_error() & binding.UQ_DEVERR_BAD_SLOT
    ok = slots.clone()
    ok[N // 2] = -1
    assert np.array_equal(cache.cpu().numpy(), _oracle_store(k, v, ok, shape))


def test_store_strided_rows_and_skipped_slots():
    N, Hk = 40, 3
    g = torch.Generator(device="cuda").manual_seed(7)
    big = torch.randn((N, 2 * Hk * 256), generator=g, device="cuda").to(torch.bfloat16)
    k = big[:, : Hk * 256].view(N, Hk, 256)            # token stride 2*Hk*D
    v = big[:, Hk * 256:].view(N, Hk, 256)
    slots = torch.arange(N, device="cuda", dtype=torch.int64) * 2
    slots[5] = -1
    slots[17] = -7
    shape = (6, 16, Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store(k, v, cache, slots)
    assert np.array_equal(cache.cpu().numpy(), _oracle_store(k, v, slots, shape))
    assert binding.uq_check_device_error() == 0


def test_store_out_of_range_slot_is_flagged_not_written():
    N, Hk = 4, 1
    k = torch.ones((N, Hk, 256), device="cuda", dtype=torch.bfloat16)
    v = torch.ones((N, Hk, 256), device="cuda", dtype=torch.bfloat16)
    slots = torch.tensor([0, 16, 1000, 3], device="cuda", dtype=torch.int64)
    cache = torch.zeros((2, 16, Hk, 272), dtype=torch.uint8, device="cuda")
    binding.uq_store(k, v, cache, slots)
    flags = binding.uq_check_device_error()
    assert flags & binding.UQ_DEVERR_BAD_SLOT
    ok = slots.clone()
    ok[2] = -1
    assert np.array_equal(cache.cpu().numpy(), _oracle_store(k, v, ok, (2, 16, Hk, 272)))
    assert binding.uq_check_device_error() == 0   # cleared by the read


def _special_rows(n_rows: int, seed: int) -> np.ndarray:
    """fp32 rows built to hit rounding ties, saturation, signed zeros, tiny
    and subnormal blocks and huge exponents."""
    rng = np.random.default_rng(seed)
    rows = rng.standard_normal((n_rows, 256)).astype(np.float32)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 6.0, 4.0], np.float32)
    for i in range(n_rows):
        kind = i % 8
        se = int(rng.integers(-100, 100))
        x = rows[i]
        if kind == 0:   # exact E2M1 ties at a random block exponent
            x[:] = rng.choice(ties, 256) * rng.choice([-1, 1], 256)
            x[::32] = 4.0          # pin each block's amax to [4, 8)
            x *= np.float32(2.0 ** se)
        elif kind == 1:  # negative values that round to zero
            x[:] = -rng.uniform(0, 0.24, 256).astype(np.float32)
            x[::32] = 4.0
        elif kind == 2:  # all-zero blocks, signed zeros
            x[:64] = 0.0
            x[64:96] = -0.0
        elif kind == 3:  # subnormal and tiny blocks
            x[:32] = np.float32(1e-39) * rng.standard_normal(32).astype(np.float32)
            x[32:64] = np.float32(1e-44)
        elif kind == 4:  # huge values near the fp32 top
            x *= np.float32(1e37)
        elif kind == 5:  # a single spike per block
            x[:] = 0.01 * x
            x[::32] = 100.0
        elif kind == 6:  # values just above/below ties
            base = rng.choice(ties, 256).astype(np.float32)
            x[:] = np.nextafter(base, np.float32(np.inf) if i % 2 else np.float32(0))
            x[::32] = 4.0
        rows[i] = x
    return rows


def test_store_rotated_f32_bit_exact_special_values():
    N, Hk = 64, 2
    kr = _special_rows(N * Hk, 1).reshape(N, Hk, 256)
    vv = _special_rows(N * Hk, 2).reshape(N, Hk, 256)
    slots = np.random.default_rng(3).permutation(8 * 16)[:N].astype(np.int64)
    shape = (8, 16, Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store_rotated_f32(torch.from_numpy(kr).cuda(), torch.from_numpy(vv).cuda(), cache,
                                 torch.from_numpy(slots).cuda())
    ref = np.zeros(shape, np.uint8)
    oracle.store_f32(kr, vv, slots, ref)
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} bytes differ"


def test_store_rotated_f32_random_rotation_bit_exact():
    """The oracle's fp64 rotation rounded to fp32, quantised by both sides."""
    N, Hk = 96, 4
    rng = np.random.default_rng(12)
    H = oracle.hadamard(256)
    k = rng.standard_normal((N, Hk, 256))
    k[..., 13] *= 30
    kr = (k @ H).astype(np.float32)
    vv = (rng.standard_normal((N, Hk, 256)) * np.exp(rng.uniform(-5, 5, (N, Hk, 1)))).astype(np.float32)
    slots = np.arange(N, dtype=np.int64)
    shape = (6, 16, Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store_rotated_f32(torch.from_numpy(kr).cuda(), torch.from_numpy(vv).cuda(), cache,
                                 torch.from_numpy(slots).cuda())
    ref = np.zeros(shape, np.uint8)
    oracle.store_f32(kr, vv, slots, ref)
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_store_full_size_bit_exact():
    """N=65536 tokens, Hk=8, 16384-page cache: every byte of the cache."""
    wl = workloads.store_workload("store")
    k, v, slots = workloads.store_inputs(wl, "cuda")
    shape = (wl.num_blocks, wl.block_size, wl.Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store(k, v, cache, slots)
    assert binding.uq_check_device_error() == 0
    got = cache.cpu().numpy()
    ref = _oracle_store(k, v, slots, shape)
    n_bad = int(np.count_nonzero(got != ref))
    assert n_bad == 0, f"{n_bad} of {got.size} bytes differ"


@pytest.mark.parametrize("Hk", [1, 3])
def test_store_bf16_special_values_bit_exact(Hk):
    """bf16 K and V built from the special fp32 rows (ties, saturation,
    signed zeros, subnormal blocks, huge exponents): V reaches the quantiser
    unrotated, K after the butterfly, both through the bf16 path's lane
    layout."""
    n_rows = 48
    kr = _special_rows(n_rows * Hk, 41)
    kr[4::8] *= np.float32(1e-3)   # keep the butterfly's sums of the huge rows finite
    k = torch.from_numpy(kr).to(torch.bfloat16).view(n_rows, Hk, 256)
    v = torch.from_numpy(_special_rows(n_rows * Hk, 42)[::-1].copy()).to(torch.bfloat16).view(n_rows, Hk, 256)
    slots = torch.from_numpy(np.random.default_rng(43).permutation(64)[:n_rows].astype(np.int64))
    shape = (4, 16, Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store(k.cuda(), v.cuda(), cache, slots.cuda())
    assert binding.uq_check_device_error() == 0
    assert np.array_equal(cache.cpu().numpy(), _oracle_store(k, v, slots, shape))
