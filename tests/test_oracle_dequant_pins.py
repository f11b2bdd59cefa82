"""Pins for the oracle's full-prefix dequantisation (uqo_full_dequant), the
bf16 prefix buffers of vllm.v1.attention.backends.ultraquant_attn,
UltraQuantAttentionImpl._ultraquant_continuation_prefill
(ultraquant_full_dequant_kv: pages -> (1, Hk, alloc_len, D), K still
rotated).  Each pin checks the oracle against something other than itself."""
from __future__ import annotations

import numpy as np
import torch

import oracle

D = 256
SB = 272
E2M1_MAGNITUDE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _mirror(cache: np.ndarray, table: np.ndarray):
    """numpy restatement of the slot layout and the dequant formula:
    element d of K is the nibble (d % 2) of byte d / 2 with the scale byte at
    256 + d / 32; V the same at 128 + d / 2 and 264 + d / 32.  Value = sign *
    magnitude * 2^(byte - 127); bf16 by torch's cast (exact: two significant
    bits, inside fp32's range)."""
    nb, bs, Hk, _ = cache.shape
    n = len(table)
    out = []
    for code_off, scale_off in ((0, 256), (128, 264)):
        slots = cache[table].reshape(n * bs, Hk, SB)            # [row, h, byte]
        d = np.arange(D)
        byte = slots[:, :, code_off + d // 2].astype(np.int64)
        code = (byte >> (4 * (d % 2))) & 15
        scale = slots[:, :, scale_off + d // 32].astype(np.int64)
        mag = E2M1_MAGNITUDE[code & 7] * np.where(code & 8, -1.0, 1.0)
        val = np.ldexp(mag, scale - 127)                         # [row, h, D] fp64
        bits = torch.from_numpy(val).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
        out.append(bits.view(np.uint16).transpose(1, 0, 2).copy())   # [h, row, D]
    return out[0], out[1]


def test_matches_numpy_mirror_on_random_bytes():
    rng = np.random.default_rng(11)
    for nb, Hk, table in ((6, 1, [0]), (9, 3, [4, 0, 8, 2]), (7, 2, [6, 6, 1])):
        cache = rng.integers(0, 256, size=(nb, 16, Hk, SB), dtype=np.uint8)
        table = np.array(table, np.int32)
        k, v, bad = oracle.full_dequant(cache, table)
        km, vm = _mirror(cache, table)
        assert bad == 0
        assert np.array_equal(k, km) and np.array_equal(v, vm)


def test_spike_row_dequantises_to_four():
    # K = 0.25 * (row i of sqrt(D) H) rotates to 4 * e_i exactly; the store
    # writes code 6 (= 4) at element i with scale byte 127 in block i / 32.
    H = oracle.hadamard(D)
    i = 77
    k = (0.25 * 16.0 * H[i]).astype(np.float32)
    kb = torch.from_numpy(k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vb = np.zeros(D, np.uint16)
    cache = np.zeros((3, 16, 1, SB), np.uint8)
    oracle.store(kb[None, None], vb[None, None], np.array([2 * 16 + 5], np.int64), cache)
    kd, vd, bad = oracle.full_dequant(cache, np.array([2], np.int32))
    expect = np.zeros(D, np.uint16)
    expect[i] = 0x4080                                          # bf16 4.0
    assert bad == 0
    assert np.array_equal(kd[0, 5], expect)
    assert not vd.any()


def test_extreme_scale_bytes_closed_form():
    # Hand-derived bf16 patterns (value = E2M1 * 2^(byte - 127)):
    #   code 1 (0.5), byte 0   -> 2^-128: subnormal, mantissa 2^-128/2^-133 = 32 -> 0x0020
    #   code 9 (-0.5), byte 0  -> -2^-128                                        -> 0x8020
    #   code 7 (6.0), byte 254 -> 1.5 * 2^129 > bf16 max -> +inf                 -> 0x7F80
    #   code 1 (0.5), byte 255 -> 2^127 (the formula read literally)              -> 0x7F00
    #   code 2 (1.0), byte 127 -> 1.0                                             -> 0x3F80
    slot = np.zeros(SB, np.uint8)
    codes = [1, 9, 7, 1, 2, 0, 0, 0]
    scales = [0, 0, 254, 255, 127, 127, 127, 127]
    for blk in range(8):
        slot[16 * blk:16 * blk + 16] = codes[blk] | (codes[blk] << 4)
        slot[256 + blk] = scales[blk]
    cache = np.zeros((1, 16, 1, SB), np.uint8)
    cache[0, 0, 0] = slot
    k, _, _ = oracle.full_dequant(cache, np.array([0], np.int32))
    expect = [0x0020, 0x8020, 0x7F80, 0x7F00, 0x3F80, 0, 0, 0]
    for blk in range(8):
        assert set(k[0, 0, 32 * blk:32 * blk + 32].tolist()) == {expect[blk]}


def test_page_permutation_invariance():
    rng = np.random.default_rng(12)
    cache = rng.integers(0, 256, size=(8, 16, 2, SB), dtype=np.uint8)
    table = np.array([5, 2, 7], np.int32)
    perm = rng.permutation(8)                                   # page x moves to perm[x]
    moved = np.empty_like(cache)
    moved[perm] = cache
    k1, v1, _ = oracle.full_dequant(cache, table)
    k2, v2, _ = oracle.full_dequant(moved, perm[table].astype(np.int32))
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)


def test_bad_page_rows_are_zero_and_counted():
    rng = np.random.default_rng(13)
    cache = rng.integers(0, 256, size=(4, 16, 2, SB), dtype=np.uint8)
    k, v, bad = oracle.full_dequant(cache, np.array([1, 9, -1, 3], np.int32))
    assert bad == 2
    assert not k[:, 16:48].any() and not v[:, 16:48].any()
    km, vm = _mirror(cache, np.array([1, 3], np.int32))
    assert np.array_equal(k[:, :16], km[:, :16]) and np.array_equal(k[:, 48:], km[:, 16:])
    assert np.array_equal(v[:, 48:], vm[:, 16:])
