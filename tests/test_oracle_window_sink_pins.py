"""Pins for the oracle's sliding window and attention sinks
(vllm.v1.attention.backends.ultraquant_attn, UltraQuantAttentionImpl:
sliding_window and sinks are handed to the unified attention with
window_size = (sliding_window - 1, 0)).  Readings checked here: a window W
keeps the last W tokens; a sink logit per query head joins the softmax
denominator only."""
from __future__ import annotations

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from test_oracle_pins import D, _bf16_bits, _fill_cache


def _decode(q, cache, perm, L, scale, splits=0, sinks=None, window=0):
    bt = np.array([perm], np.int32)
    return oracle.decode(_bf16_bits(q)[None], cache, bt, np.array([L], np.int32), scale,
                         splits=splits, nthreads=2, sinks=sinks, window=window)[0]


def _random_seq(seed, L, Hk):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((L, Hk, D)).astype(np.float32)
    v = rng.standard_normal((L, Hk, D)).astype(np.float32)
    return rng, k, v


def test_window_at_least_length_changes_nothing():
    rng, k, v = _random_seq(30, 45, 1)
    perm = [2, 0, 1]
    cache = _fill_cache(k, v, 1, perm)
    q = rng.standard_normal((8, D)).astype(np.float32)
    ref = _decode(q, cache, perm, 45, 1 / 16)
    for w in (45, 46, 10_000):
        assert np.array_equal(_decode(q, cache, perm, 45, 1 / 16, window=w), ref)


def test_window_one_returns_the_last_value():
    rng, k, v = _random_seq(31, 37, 1)
    perm = [1, 2, 0]
    cache = _fill_cache(k, v, 1, perm)
    out = _decode(rng.standard_normal((8, D)).astype(np.float32), cache, perm, 37, 0.3, window=1)
    _, vlast = oracle.dequant_slot(cache[perm[36 // 16], 36 % 16, 0])
    for r in range(8):
        assert np.array_equal(out[r], vlast)


@pytest.mark.parametrize("w", [2, 15, 16, 17, 40])
def test_window_equals_decoding_only_the_last_tokens(w):
    """The window's tokens stored again as a short sequence of their own."""
    L = 70
    rng, k, v = _random_seq(32 + w, L, 2)
    perm = list(rng.permutation(5))
    cache = _fill_cache(k, v, 2, perm)
    q = rng.standard_normal((16, D)).astype(np.float32)
    got = _decode(q, cache, perm, L, 1 / 16, window=w)
    short_perm = list(range((w + 15) // 16))
    short = _fill_cache(k[L - w:], v[L - w:], 2, short_perm)
    assert np.array_equal(got, _decode(q, short, short_perm, w, 1 / 16))


def test_sink_with_equal_keys_closed_form():
    """All scores equal s: out = mean(v) * L e^s / (L e^s + e^z); z = s + ln L halves it."""
    L, Hq = 24, 8
    rng = np.random.default_rng(33)
    k1 = rng.standard_normal(D).astype(np.float32)
    k = np.broadcast_to(k1, (L, 1, D)).copy()
    v = rng.standard_normal((L, 1, D)).astype(np.float32)
    perm = [0, 1]
    cache = _fill_cache(k, v, 1, perm)
    q = rng.standard_normal((Hq, D)).astype(np.float32)
    scale = 0.2
    plain = _decode(q, cache, perm, L, scale)
    khat = oracle.dequant_slot(cache[0, 0, 0])[0]
    s = np.array([scale * (oracle.query_prime(_bf16_bits(q[r])) @ khat) for r in range(Hq)])
    z = s + np.log(L)
    out = _decode(q, cache, perm, L, scale, sinks=z)
    vhat = np.stack([oracle.dequant_slot(cache[t // 16, t % 16, 0])[1] for t in range(L)]).mean(0)
    for r in range(Hq):
        assert np.abs(plain[r] - vhat).max() <= 1e-12
        assert np.abs(out[r] - 0.5 * vhat).max() <= 1e-12


def test_sink_at_minus_infinity_changes_nothing():
    rng, k, v = _random_seq(34, 50, 1)
    perm = [3, 1, 0, 2]
    cache = _fill_cache(k, v, 1, perm)
    q = rng.standard_normal((8, D)).astype(np.float32)
    ref = _decode(q, cache, perm, 50, 1 / 16)
    assert np.array_equal(_decode(q, cache, perm, 50, 1 / 16, sinks=np.full(8, -np.inf)), ref)


@pytest.mark.parametrize("L,w", [(33, 0), (100, 37), (257, 16), (5, 3)])
def test_split_then_merge_with_window_and_sinks(L, w):
    rng, k, v = _random_seq(35 + L, L, 1)
    perm = list(rng.permutation((L + 15) // 16))
    cache = _fill_cache(k, v, 1, perm)
    q = rng.standard_normal((8, D)).astype(np.float32) * 3
    sinks = rng.standard_normal(8) * 4
    ref = _decode(q, cache, perm, L, 1 / 16, sinks=sinks, window=w)
    for S in (1, 2, 7, 32):
        got = _decode(q, cache, perm, L, 1 / 16, splits=S, sinks=sinks, window=w)
        assert np.abs(got - ref).max() <= 1e-12


def test_brute_force_window_and_sinks():
    """Independent restatement: scipy Hadamard, numpy LUT, numpy softmax over
    the window with the sink column dropped."""
    lut = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    H = scipy.linalg.hadamard(D) / 16.0
    L, Hk, Hq, w = 61, 2, 12, 23
    rng, k, v = _random_seq(36, L, Hk)
    perm = list(rng.permutation(4))
    cache = _fill_cache(k, v, Hk, perm)
    qb = _bf16_bits(rng.standard_normal((Hq, D)).astype(np.float32))
    sinks = rng.standard_normal(Hq) * 3
    got = oracle.decode(qb[None], cache, np.array([perm], np.int32), np.array([L], np.int32), 0.1,
                        nthreads=2, sinks=sinks, window=w)[0]
    t = np.arange(L - w, L)
    slots = cache[np.array(perm)[t // 16], t % 16]
    lo, hi = slots[..., :256] & 15, slots[..., :256] >> 4
    codes = np.stack([lo, hi], -1).reshape(w, Hk, 512)
    kh = lut[codes[..., :256]] * np.exp2(np.repeat(slots[..., 256:264].astype(np.float64) - 127, 32, -1))
    vh = lut[codes[..., 256:]] * np.exp2(np.repeat(slots[..., 264:272].astype(np.float64) - 127, 32, -1))
    for r in range(Hq):
        qr = (oracle.bf16_bits_to_f64(qb[r]) @ H).astype(np.float32)
        qp = torch.from_numpy(qr).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        s = 0.1 * (kh[:, r // 6] @ qp)
        m = s.max()
        p = np.exp(s - m)
        ref = (p[:, None] * vh[:, r // 6]).sum(0) / (p.sum() + np.exp(sinks[r] - m))
        assert np.abs(got[r] - ref).max() <= 1e-12
