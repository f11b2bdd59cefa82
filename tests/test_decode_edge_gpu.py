"""GPU parity of decode against the fp64 oracle on the method's extreme cases:
the places where the CUDA arithmetic departs from the oracle's.

The CUDA decode runs the tensor-core products on f16 operands: each token's
largest UE8M0 block exponent is factored out and the other blocks are scaled
relative to it (an exact power of two over a span of 2^27); K blocks further
below are added back by an exact fp32 path.  The query is rounded through
E4M3 with saturation (flydsl_ultraquant_decode, the Q prologue's "always
apply the E4M3 haircut"), and the FP4 values are the E2M1 table times
2^(byte - 127) (the same page's _fp4_value_lut).  Each test builds a cache
with uq_store_rotated_f32 (and, for scale bytes the store never writes, by
editing cache bytes), checks that cache byte for byte against the oracle's
own packing, and compares uq_decode / uq_decode_ex with oracle.decode at
max-abs 1e-2 and relative L2 5e-3.

Rows whose exact output exceeds 1 in magnitude (V at fp32's top end) are
compared after dividing both sides by the row's largest exact element: a
bf16 output near 2^127 has a quantum of 2^119, so no implementation can meet
an absolute 1e-2 there; the relative form is the same bound in units of the
output.  Scores must stay inside fp32 (|scale * q'.k| < 2^127), as for any
fp32 accumulation: K blocks near fp32's top are therefore met only by query
rows that are zero on those blocks.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads

from _util import compare, lib

pytestmark = pytest.mark.gpu

D = 256
GROUPS = [(8, 1), (12, 2), (32, 2)]     # query heads per kv head: 8, 6, 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    assert binding.uq_check_device_error() == 0


def _layout(lens, Hq, Hk, seed, splits=5):
    lens = np.asarray(lens, np.int32)
    max_blocks = int((lens.max() + 15) // 16)
    return workloads.make_decode_workload("edge", len(lens), Hq, Hk, lens, max_blocks, splits,
                                          seed=seed, spare_blocks=2)


def _fill(wl, kr: np.ndarray, vv: np.ndarray):
    """Store fp32 rotated K and V [sum(L), Hk, D] (sequence after sequence)
    with uq_store_rotated_f32 and with the oracle; the two caches must agree."""
    slots = np.concatenate([workloads.sequence_slots(wl, b) for b in range(wl.B)])
    shape = (wl.num_blocks, wl.block_size, wl.Hk, 272)
    cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    binding.uq_store_rotated_f32(torch.from_numpy(np.ascontiguousarray(kr, np.float32)).cuda(),
                                 torch.from_numpy(np.ascontiguousarray(vv, np.float32)).cuda(), cache,
                                 torch.from_numpy(slots).cuda())
    ref = np.zeros(shape, np.uint8)
    oracle.store_f32(kr, vv, slots, ref)
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} cache bytes differ"
    assert binding.uq_check_device_error() == 0
    return ref


def _query_from_prime(qp: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of q = q' H for a target q' of small integers: every
    entry of q is a multiple of 1/16 of magnitude <= 16, exact in bf16, and
    the rotation maps it back to q' exactly (H = H^T, H H = I)."""
    q = qp @ oracle.hadamard(D)
    bits = oracle.bf16_round_array(q)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), q), "q is not exact in bf16"
    flat_b, flat_p = bits.reshape(-1, D), qp.reshape(-1, D)
    for i in range(0, flat_b.shape[0], max(1, flat_b.shape[0] // 5)):
        assert np.array_equal(oracle.query_prime(flat_b[i]), flat_p[i])
    return bits


def _decode(wl, cache_np, q_bits, sinks=None, window=0):
    dev = "cuda"
    cache = torch.from_numpy(cache_np).to(dev)
    q = torch.from_numpy(q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, D, wl.splits), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.B, wl.Hq, D), dtype=torch.bfloat16, device=dev)
    if sinks is None and window == 0:
        binding.uq_decode(q, cache, bt, sl, wl.scale, wl.splits, ws, out)
    else:
        sk = None if sinks is None else torch.from_numpy(np.asarray(sinks, np.float32)).to(dev)
        binding.uq_decode_ex(q, cache, bt, sl, wl.scale, sk, window, wl.splits, ws, out)
    assert binding.uq_check_device_error() == 0
    return out


def _oracle(wl, cache_np, q_bits, sinks=None, window=0):
    return oracle.decode(q_bits, cache_np, wl.block_table, wl.seq_lens, wl.scale,
                         sinks=sinks, window=window)


def _compare_scaled(got: torch.Tensor, ref: np.ndarray):
    """The decode bound on each row divided by max(1, its largest exact |value|)."""
    g = got.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    s = np.maximum(1.0, np.abs(ref).max(axis=-1, keepdims=True))
    assert np.isfinite(g).all(), "non-finite GPU output"
    compare(torch.from_numpy(g / s), ref / s)


def _rows(rng, n_tok, Hk, scale=1.0):
    return (rng.standard_normal((n_tok, Hk, D)) * scale).astype(np.float32)


# --------------------------------------------------------------------------- #
# (a) block exponent spreads beyond the f16 span of one token                  #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("Hq,Hk", GROUPS)
@pytest.mark.parametrize("big_log2,n_big", [(20, 1), (20, 7), (27, 1), (28, 3), (60, 1), (100, 7)])
@pytest.mark.parametrize("window", [0, 50])
def test_k_block_spread(Hq, Hk, big_log2, n_big, window):
    """Per token, n_big K blocks at 2^big_log2 and the rest at 2^0, and query
    rows that are zero on the big blocks: the scores come only from the
    small blocks, so a path that dropped them would give a uniform softmax.
    Spreads of 2^28 and more go through the exact fp32 path.  (Rows that
    also see the big blocks have scores near 2^big_log2 whose top values tie
    on the E2M1 lattice and are told apart by O(1) terms, below fp32's
    resolution there for any fp32 accumulation; the dominant-token test
    below covers large scores where the answer is well conditioned.)"""
    rng = np.random.default_rng(1000 + big_log2 + 3 * n_big + Hq)
    lens = [1, 37, 300, 16]
    wl = _layout(lens, Hq, Hk, seed=11 + n_big)
    n = int(np.sum(lens))
    big = [0] if n_big == 1 else [b for b in range(8) if b != 3][:n_big]
    kr = _rows(rng, n, Hk)
    for blk in big:
        kr[:, :, 32 * blk:32 * blk + 32] *= np.float32(2.0 ** big_log2)
    vv = _rows(rng, n, Hk)
    ref_cache = _fill(wl, kr, vv)
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    for blk in big:
        qp[..., 32 * blk:32 * blk + 32] = 0.0
    q_bits = _query_from_prime(qp)
    out = _decode(wl, ref_cache, q_bits, window=window)
    compare(out, _oracle(wl, ref_cache, q_bits, window=window))


@pytest.mark.parametrize("Hq,Hk", GROUPS)
@pytest.mark.parametrize("every", [37, 400])
def test_k_block_spread_on_some_tokens(Hq, Hk, every):
    """Only every `every`-th token carries a K block at 2^40 (query rows zero
    there): the units holding one are redone exactly, the others keep the
    tensor-core result, and both kinds sit in one batch."""
    rng = np.random.default_rng(1200 + every + Hq)
    lens = [3, 700, 1500, 64]
    wl = _layout(lens, Hq, Hk, seed=13, splits=6)
    n = int(np.sum(lens))
    kr = _rows(rng, n, Hk)
    kr[5::every, :, 96:128] *= np.float32(2.0 ** 40)
    vv = _rows(rng, n, Hk)
    ref_cache = _fill(wl, kr, vv)
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    qp[..., 96:128] = 0.0
    q_bits = _query_from_prime(qp)
    out = _decode(wl, ref_cache, q_bits)
    compare(out, _oracle(wl, ref_cache, q_bits))


@pytest.mark.parametrize("Hq,Hk", GROUPS)
def test_k_block_spread_under_graph_replay(Hq, Hk):
    """One captured decode replayed with new lengths over a cache whose far
    K blocks (2^40, query rows zero there) sit only from token 400 on: the
    exact pass's list is rebuilt on every replay, from empty (all lengths
    below 400) to every unit of the long sequences, and each replay matches
    both the oracle and an eager call."""
    rng = np.random.default_rng(1250 + Hq)
    lens = [3, 700, 1500, 64]
    wl = _layout(lens, Hq, Hk, seed=15, splits=6)
    n = int(np.sum(lens))
    kr = _rows(rng, n, Hk)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    for b, L in enumerate(lens):
        kr[starts[b] + 400:starts[b] + L, :, 224:256] *= np.float32(2.0 ** 40)
    vv = _rows(rng, n, Hk)
    ref_cache = _fill(wl, kr, vv)
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    qp[..., 224:256] = 0.0
    q_bits = _query_from_prime(qp)
    dev = "cuda"
    cache = torch.from_numpy(ref_cache).to(dev)
    q = torch.from_numpy(q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    bt = torch.from_numpy(wl.block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, D, wl.splits), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.B, wl.Hq, D), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        binding.uq_decode(q, cache, bt, sl, wl.scale, wl.splits, ws, out)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        binding.uq_decode(q, cache, bt, sl, wl.scale, wl.splits, ws, out)
    for new_lens in ([3, 700, 1500, 64], [3, 399, 390, 64], [0, 401, 1500, 0], [3, 700, 1500, 64]):
        nl = np.array(new_lens, np.int32)
        sl.copy_(torch.from_numpy(nl))
        graph.replay()
        torch.cuda.synchronize()
        assert binding.uq_check_device_error() == 0
        ref = oracle.decode(q_bits, ref_cache, wl.block_table, nl, wl.scale)
        compare(out, ref)
        eager = torch.empty_like(out)
        binding.uq_decode(q, cache, bt, torch.from_numpy(nl).to(dev), wl.scale, wl.splits, ws, eager)
        assert torch.equal(out, eager)


@pytest.mark.parametrize("Hq,Hk,cached,q_len,block_size", [
    (8, 1, 300, 5, 16),
    (12, 2, 95, 3, 64),
    (32, 2, 40, 4, 32),
])
def test_k_block_spread_multi_query(Hq, Hk, cached, q_len, block_size):
    """K blocks at 2^40 on every token (query rows zero there) through the
    multi-query entry and pages of more than 16 tokens: the exact pass redoes
    the units with each chunk row's own causal range."""
    rng = np.random.default_rng(1300 + cached + block_size)
    L = cached + q_len
    P = (L + block_size - 1) // block_size
    S = 4
    wl = workloads.make_decode_workload("edge_mq", 1, Hq, Hk, np.array([L]), P + 1, S, seed=14,
                                        spare_blocks=2, block_size=block_size)
    kr = _rows(rng, L, Hk)
    kr[:, :, 0:32] *= np.float32(2.0 ** 40)
    vv = _rows(rng, L, Hk)
    ref_cache = _fill(wl, kr, vv)
    qp = rng.integers(-2, 3, size=(q_len, Hq, D)).astype(np.float64)
    qp[..., 0:32] = 0.0
    q_bits = _query_from_prime(qp)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    cache = torch.from_numpy(ref_cache).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).cuda()
    ws = torch.empty(binding.uq_decode_workspace_bytes(q_len, Hq, D, S), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out)
    assert binding.uq_check_device_error() == 0
    table = np.tile(wl.block_table[0], (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    compare(out, oracle.decode(q_bits, ref_cache, table, lens, wl.scale))


@pytest.mark.parametrize("Hq,Hk", GROUPS)
@pytest.mark.parametrize("big_log2", [20, 60])
def test_one_dominant_token_with_huge_scores(Hq, Hk, big_log2):
    """One token per sequence carries a K block at 2^big_log2 aligned with
    every query row, another the same block negated; all other tokens are
    ordinary.  Scores reach 2^big_log2 / 16, the softmax is one-hot on the
    first token, and the output is its V row."""
    rng = np.random.default_rng(1500 + big_log2 + Hq)
    lens = [3, 90, 200]
    wl = _layout(lens, Hq, Hk, seed=19)
    n = int(np.sum(lens))
    kr = _rows(rng, n, Hk)
    vv = _rows(rng, n, Hk)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    for b, s0 in enumerate(starts):
        hot, cold = s0 + (7 * b + 1) % lens[b], s0 + (11 * b + 2) % lens[b]
        kr[hot, :, 64:96] = np.float32(2.0 ** big_log2)
        if cold != hot:
            kr[cold, :, 64:96] = -np.float32(2.0 ** big_log2)
    ref_cache = _fill(wl, kr, vv)
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    qp[..., 64:96] = 1.0
    q_bits = _query_from_prime(qp)
    out = _decode(wl, ref_cache, q_bits)
    compare(out, _oracle(wl, ref_cache, q_bits))


@pytest.mark.parametrize("Hq,Hk", GROUPS)
@pytest.mark.parametrize("big_log2,small_log2", [(0, -20), (0, -40), (20, 0)])
def test_v_block_spread(Hq, Hk, big_log2, small_log2):
    """Per token, one V block at 2^big_log2 and the rest at 2^small_log2; K
    ordinary.  Outputs of the large-V case are compared in units of the row."""
    rng = np.random.default_rng(2000 + big_log2 - small_log2 + Hq)
    lens = [5, 129, 260]
    wl = _layout(lens, Hq, Hk, seed=12)
    n = int(np.sum(lens))
    kr = _rows(rng, n, Hk)
    vv = _rows(rng, n, Hk)
    for blk in range(8):
        vv[:, :, 32 * blk:32 * blk + 32] *= np.float32(2.0 ** (big_log2 if blk == 2 else small_log2))
    ref_cache = _fill(wl, kr, vv)
    q_bits = oracle.bf16_round_array(rng.standard_normal((wl.B, Hq, D)))
    out = _decode(wl, ref_cache, q_bits)
    _compare_scaled(out, _oracle(wl, ref_cache, q_bits))


# --------------------------------------------------------------------------- #
# (b) scale bytes at both ends                                                 #
# --------------------------------------------------------------------------- #

def _amax_rows(rng, n, Hk, amax_of_block):
    """Rows whose block b has amax exactly amax_of_block(b) (values below it
    drawn uniformly, one element pinned to +-amax)."""
    x = np.empty((n, Hk, D), np.float32)
    for blk in range(8):
        a = amax_of_block(blk)
        x[:, :, 32 * blk:32 * blk + 32] = (rng.uniform(-1, 1, (n, Hk, 32)) * a).astype(np.float32)
        x[:, :, 32 * blk] = np.float32(a) * rng.choice([-1, 1], (n, Hk)).astype(np.float32)
    return x


@pytest.mark.parametrize("Hq,Hk", GROUPS)
def test_tiny_scale_bytes_0_and_1(Hq, Hk):
    """K and V blocks whose amax gives UE8M0 bytes 0 and 1 (values near and
    below fp32's smallest normal), mixed with ordinary tokens."""
    rng = np.random.default_rng(3000 + Hq)
    lens = [40, 17, 200]
    wl = _layout(lens, Hq, Hk, seed=13)
    n = int(np.sum(lens))
    tiny = _amax_rows(rng, n, Hk, lambda b: 2.0 ** -125 if b % 2 else 2.0 ** -124)  # bytes 0, 1
    kr = _rows(rng, n, Hk)
    vv = _rows(rng, n, Hk)
    sel_k = rng.random(n) < 0.5
    sel_v = rng.random(n) < 0.5
    kr[sel_k] = tiny[sel_k]
    vv[sel_v] = tiny[::-1][sel_v]
    ref_cache = _fill(wl, kr, vv)
    k_bytes = ref_cache[..., 256:264]
    assert (k_bytes == 0).any() and (k_bytes == 1).any()
    q_bits = oracle.bf16_round_array(rng.standard_normal((wl.B, Hq, D)))
    out = _decode(wl, ref_cache, q_bits)
    compare(out, _oracle(wl, ref_cache, q_bits))


@pytest.mark.parametrize("Hq,Hk", GROUPS)
def test_top_scale_bytes_from_fp32_ends(Hq, Hk):
    """V blocks near fp32's largest values (byte 252, the top the store can
    reach from fp32) in some tokens, and K blocks there met by query rows that
    are zero on them (their other blocks ordinary: a spread of 2^125)."""
    rng = np.random.default_rng(4000 + Hq)
    lens = [33, 150, 2]
    wl = _layout(lens, Hq, Hk, seed=14)
    n = int(np.sum(lens))
    kr = _rows(rng, n, Hk)
    vv = _rows(rng, n, Hk)
    huge_k = rng.random(n) < 0.4
    kr[huge_k, :, 64:96] = (rng.uniform(-1, 1, (int(huge_k.sum()), Hk, 32)) * 3e38).astype(np.float32)
    huge_v = rng.random(n) < 0.3
    vv[huge_v, :, 160:192] = (rng.uniform(-1, 1, (int(huge_v.sum()), Hk, 32)) * 3e38).astype(np.float32)
    ref_cache = _fill(wl, kr, vv)
    assert ref_cache[..., 256:272].max() == 252
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    qp[..., 64:96] = 0.0
    q_bits = _query_from_prime(qp)
    out = _decode(wl, ref_cache, q_bits)
    _compare_scaled(out, _oracle(wl, ref_cache, q_bits))


@pytest.mark.parametrize("Hq,Hk", GROUPS)
def test_scale_bytes_253_254_written_into_the_cache(Hq, Hk):
    """Bytes 253 and 254 never come out of the store; a cache edited to hold
    them must decode like the oracle: V blocks with codes of magnitude <= 1.5
    (so 1.5 * 2^127 stays finite), K blocks met by query rows zero on them."""
    rng = np.random.default_rng(5000 + Hq)
    lens = [60, 21]
    wl = _layout(lens, Hq, Hk, seed=15)
    n = int(np.sum(lens))
    cache = _fill(wl, _rows(rng, n, Hk), _rows(rng, n, Hk))
    slots = np.concatenate([workloads.sequence_slots(wl, b) for b in range(wl.B)])
    flat = cache.reshape(-1, wl.Hk, 272)
    for i, s in enumerate(slots):
        for h in range(wl.Hk):
            if rng.random() < 0.35:                     # V block 6 at 2^126 or 2^127
                flat[s, h, 264 + 6] = 253 + (i + h) % 2
                codes = rng.integers(0, 4, 32) | (rng.integers(0, 2, 32) << 3)   # |value| <= 1.5
                flat[s, h, 128 + 96:128 + 112] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
            if rng.random() < 0.35:                     # K block 1 at 2^126 or 2^127
                flat[s, h, 256 + 1] = 254 - (i + h) % 2
    qp = rng.integers(-2, 3, size=(wl.B, Hq, D)).astype(np.float64)
    qp[..., 32:64] = 0.0
    q_bits = _query_from_prime(qp)
    out = _decode(wl, cache, q_bits)
    _compare_scaled(out, _oracle(wl, cache, q_bits))


# --------------------------------------------------------------------------- #
# (c) E4M3 saturation of the rotated query                                     #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("Hq,Hk", GROUPS)
def test_query_rotation_saturates_e4m3(Hq, Hk):
    """q = 64 * ones rotates to 1024 * e_0, which saturates to 448; large
    random queries saturate in many head dims.  q' is checked against the
    oracle's haircut first."""
    rng = np.random.default_rng(6000 + Hq)
    lens = [19, 333]
    wl = _layout(lens, Hq, Hk, seed=16)
    n = int(np.sum(lens))
    ref_cache = _fill(wl, _rows(rng, n, Hk, 0.05), _rows(rng, n, Hk))
    q = rng.standard_normal((wl.B, Hq, D)) * 300.0
    q[:, 0] = 64.0
    q_bits = oracle.bf16_round_array(q)
    qp0 = oracle.query_prime(q_bits[0, 0])
    assert qp0[0] == 448.0 and not qp0[1:].any()
    assert (np.abs(oracle.query_prime(q_bits[1, 1])) == 448.0).sum() > 10
    out = _decode(wl, ref_cache, q_bits)
    compare(out, _oracle(wl, ref_cache, q_bits))


# --------------------------------------------------------------------------- #
# (d) sinks at -inf and far above every score                                  #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("Hq,Hk", GROUPS)
@pytest.mark.parametrize("kind", ["neg_inf", "far_above", "mixed"])
def test_extreme_sinks(Hq, Hk, kind):
    rng = np.random.default_rng(7000 + Hq)
    lens = [1, 90, 700]
    wl = _layout(lens, Hq, Hk, seed=17)
    n = int(np.sum(lens))
    ref_cache = _fill(wl, _rows(rng, n, Hk), _rows(rng, n, Hk))
    q_bits = oracle.bf16_round_array(rng.standard_normal((wl.B, Hq, D)))
    if kind == "neg_inf":
        sinks = np.full(Hq, -np.inf)
    elif kind == "far_above":
        sinks = np.full(Hq, 1.0e4)
    else:
        sinks = np.where(np.arange(Hq) % 2 == 0, -np.inf, 30.0)
        sinks[1] = 2.0
    for window in (0, 64):
        out = _decode(wl, ref_cache, q_bits, sinks=sinks, window=window)
        ref = _oracle(wl, ref_cache, q_bits, sinks=sinks, window=window)
        compare(out, ref)
        if kind == "neg_inf":   # a sink at -inf changes nothing
            plain = _decode(wl, ref_cache, q_bits, window=window)
            assert torch.equal(out, plain)
