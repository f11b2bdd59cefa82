"""Seeded synthetic workloads for the store and decode paths.

This module draws random inputs only: sequence lengths, page tables, bf16
query/K/V tensors and slot mappings.  It contains none of the method's
arithmetic (no rotation, quantisation or attention), so the CUDA path and the
CPU oracle can both be fed from it without sharing any of the computation.

Recipe (every workload; the pages measure on no public dataset, so these
synthetic draws stand in for real traffic):
  * sequence metadata: numpy ``default_rng(seed)``; pages of all sequences
    are a random permutation of ``arange(num_blocks)`` handed out in order,
    so consecutive pages of a sequence are scattered in the cache; unused
    block-table entries are 0.
  * tensors: torch ``randn`` (fp32) rounded to bf16, from a
    ``torch.Generator`` on the requested device seeded per sequence
    (``seed * 1_000_003 + b + 1``) so one sequence can be regenerated alone.
  * outlier-K workload: 4 channels per kv head drawn once from the seed,
    multiplied by 20 in every token of K.
  * full-dequant workload: one sequence of 32768 tokens (2048 pages) and 8 kv
    heads, its K/V drawn like a decode workload's and written with uq_store;
    pages are a random permutation of the cache.
  * store workload: K and V ~ N(0, 1) with independent Bernoulli(0.01)
    masks multiplying entries by 50; slots are the first N of a random
    permutation of all num_blocks * block_size slots.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEAD_DIM = 256
BLOCK_SIZE = 16


@dataclasses.dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hk: int
    splits: int
    scale: float
    seed: int
    seq_lens: np.ndarray          # int32 [B]
    max_blocks: int               # block-table width
    block_table: np.ndarray       # int32 [B, max_blocks]
    num_blocks: int
    outlier_channels: np.ndarray | None = None   # int [Hk, 4]
    outlier_factor: float = 20.0
    D: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    graph_replay: bool = False

    @property
    def QG(self) -> int:
        return self.Hq // self.Hk

    def kv_bytes(self) -> int:
        """Packed-cache bytes a decode pass reads: sum(L) * Hk * 272."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hk * (self.D + self.D // 16)

    def algorithmic_bytes(self) -> int:
        """Packed KV read + bf16 query read + bf16 output written."""
        return self.kv_bytes() + 2 * self.B * self.Hq * self.D * 2


def _pages(seq_lens: np.ndarray, bs: int) -> np.ndarray:
    return (seq_lens.astype(np.int64) + bs - 1) // bs


def make_decode_workload(name: str, B: int, Hq: int, Hk: int, seq_lens: np.ndarray,
                         max_blocks: int, splits: int, seed: int, scale: float = 1.0 / 16,
                         outliers: bool = False, graph_replay: bool = False,
                         spare_blocks: int = 0, block_size: int = BLOCK_SIZE) -> DecodeWorkload:
    rng = np.random.default_rng(seed + 7919)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    pages = _pages(seq_lens, block_size)
    assert int(pages.max(initial=0)) <= max_blocks
    num_blocks = int(pages.sum()) + spare_blocks
    perm = rng.permutation(max(num_blocks, 1)).astype(np.int32)
    bt = np.zeros((B, max_blocks), dtype=np.int32)
    pos = 0
    for b in range(B):
        n = int(pages[b])
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    oc = None
    if outliers:
        crng = np.random.default_rng(seed + 104729)
        oc = np.stack([crng.choice(HEAD_DIM, 4, replace=False) for _ in range(Hk)])
    return DecodeWorkload(name, B, Hq, Hk, splits, scale, seed, seq_lens, max_blocks, bt,
                          max(num_blocks, 1), oc, graph_replay=graph_replay, block_size=block_size)


def decode_workload(name: str) -> DecodeWorkload:
    """The four decode workloads.

    tiny          B=1,   Hq=8,  Hk=1 (GQA 8),  L=512, 32 pages, S=4, seed 0
    batch         B=32,  Hq=32, Hk=4 (GQA 8),  L ~ U{1024..8192},  S=32, seed 1
    outlier_long  B=64,  Hq=48, Hk=8 (GQA 6),  L ~ U{16384..32768}, S=32, seed 2,
                  outlier K channels
    skewed        B=128, Hq=64, Hk=4 (GQA 16), L = floor(exp(U(ln 128, ln 131072))),
                  max_model_len 131072, S=32, seed 3, CUDA-graph replay
    outlier_ncu   B=16, Hq=48, Hk=8, L=16384 each, outlier K: the outlier shape at a
                  size a full ncu capture can replay (570 MB of cache)
    skewed_ncu    B=16, Hq=64, Hk=4 (GQA 16), L=16384 each: the skewed head shape
                  for a full ncu capture (285 MB of cache)
    All use D=256, block_size=16, scale=1/16, bf16 q/K/V ~ N(0,1).
    """
    if name == "tiny":
        return make_decode_workload("tiny", 1, 8, 1, np.array([512]), 32, 4, seed=0)
    if name == "batch":
        rng = np.random.default_rng(1)
        lens = rng.integers(1024, 8192 + 1, size=32)
        return make_decode_workload("batch", 32, 32, 4, lens, 8192 // BLOCK_SIZE, 32, seed=1)
    if name == "outlier_long":
        rng = np.random.default_rng(2)
        lens = rng.integers(16384, 32768 + 1, size=64)
        return make_decode_workload("outlier_long", 64, 48, 8, lens, 32768 // BLOCK_SIZE, 32,
                                    seed=2, outliers=True)
    if name == "outlier_ncu":
        # the outlier workload's shape at 16 sequences of 16384 tokens (570 MB
        # of cache, above L2, small enough for a full ncu capture)
        return make_decode_workload("outlier_ncu", 16, 48, 8, np.full(16, 16384), 16384 // BLOCK_SIZE,
                                    32, seed=2, outliers=True)
    if name == "skewed_ncu":
        # the skewed workload's GQA-16 head shape at 16 sequences of 16384
        # tokens (285 MB of cache, above L2, small enough for a full ncu capture)
        return make_decode_workload("skewed_ncu", 16, 64, 4, np.full(16, 16384), 16384 // BLOCK_SIZE,
                                    32, seed=3)
    if name == "skewed":
        rng = np.random.default_rng(3)
        lens = np.floor(np.exp(rng.uniform(math.log(128), math.log(131072), size=128)))
        lens = np.minimum(lens, 131072).astype(np.int32)
        return make_decode_workload("skewed", 128, 64, 4, lens, 131072 // BLOCK_SIZE, 32,
                                    seed=3, graph_replay=True)
    raise KeyError(name)


DECODE_WORKLOADS = ("tiny", "batch", "outlier_long", "skewed", "outlier_ncu", "skewed_ncu")


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def sequence_kv(wl: DecodeWorkload, b: int, device="cpu"):
    """bf16 K, V [L_b, Hk, D] of sequence b (deterministic per (seed, b, device type))."""
    L = int(wl.seq_lens[b])
    gen = _gen(device, wl.seed * 1_000_003 + b + 1)
    k = torch.randn((L, wl.Hk, wl.D), generator=gen, device=device, dtype=torch.float32)
    v = torch.randn((L, wl.Hk, wl.D), generator=gen, device=device, dtype=torch.float32)
    if wl.outlier_channels is not None:
        for h in range(wl.Hk):
            idx = torch.as_tensor(wl.outlier_channels[h], device=device, dtype=torch.long)
            k[:, h, idx] *= wl.outlier_factor
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def sequence_slots(wl: DecodeWorkload, b: int) -> np.ndarray:
    """int64 slot of every token of sequence b (page * block_size + offset)."""
    L = int(wl.seq_lens[b])
    t = np.arange(L, dtype=np.int64)
    return wl.block_table[b, t // wl.block_size].astype(np.int64) * wl.block_size + t % wl.block_size


def query(wl: DecodeWorkload, device="cpu", step: int = 0) -> torch.Tensor:
    """bf16 query [B, Hq, D] for decode step `step`."""
    gen = _gen(device, wl.seed * 1_000_003 + 999_983 + 7 * step)
    return _randn_bf16((wl.B, wl.Hq, wl.D), gen, device)


def chunk_query(wl: DecodeWorkload, q_len: int, device="cpu", step: int = 0) -> torch.Tensor:
    """bf16 query [q_len, Hq, D] of a continuation chunk of sequence 0."""
    gen = _gen(device, wl.seed * 1_000_003 + 333_331 + 7 * step)
    return _randn_bf16((q_len, wl.Hq, wl.D), gen, device)


def new_token_kv(wl: DecodeWorkload, device="cpu", step: int = 0):
    """bf16 K, V [B, Hk, D] of the token each sequence appends at a decode step."""
    gen = _gen(device, wl.seed * 1_000_003 + 499_979 + 7 * step)
    k = torch.randn((wl.B, wl.Hk, wl.D), generator=gen, device=device, dtype=torch.float32)
    v = torch.randn((wl.B, wl.Hk, wl.D), generator=gen, device=device, dtype=torch.float32)
    if wl.outlier_channels is not None:
        for h in range(wl.Hk):
            idx = torch.as_tensor(wl.outlier_channels[h], device=device, dtype=torch.long)
            k[:, h, idx] *= wl.outlier_factor
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def last_slots(wl: DecodeWorkload) -> np.ndarray:
    """Slot of each sequence's last token (where a decode step writes its new K/V)."""
    L = wl.seq_lens.astype(np.int64)
    t = np.maximum(L - 1, 0)
    slots = wl.block_table[np.arange(wl.B), t // wl.block_size].astype(np.int64) * wl.block_size + t % wl.block_size
    return np.where(L > 0, slots, -1)


@dataclasses.dataclass
class StoreWorkload:
    name: str
    N: int
    Hk: int
    num_blocks: int
    seed: int
    outlier_p: float = 0.01
    outlier_factor: float = 50.0
    D: int = HEAD_DIM
    block_size: int = BLOCK_SIZE

    def algorithmic_bytes(self) -> int:
        """bf16 K and V read, 272-byte slots written, int64 slot ids read."""
        return self.N * self.Hk * (2 * self.D * 2 + self.D + self.D // 16) + 8 * self.N


def store_workload(name: str = "store") -> StoreWorkload:
    """N=65536 new tokens, Hk=8, into a 16384-page cache (block_size 16), seed 4."""
    if name == "store":
        return StoreWorkload("store", 65536, 8, 16384, seed=4)
    if name == "store_small":
        return StoreWorkload("store_small", 1000, 3, 80, seed=5)
    raise KeyError(name)


def store_inputs(wl: StoreWorkload, device="cpu"):
    """bf16 K, V [N, Hk, D] with outliers and int64 slot_mapping [N]."""
    gen = _gen(device, wl.seed * 1_000_003 + 1)
    shape = (wl.N, wl.Hk, wl.D)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    km = torch.rand(shape, generator=gen, device=device) < wl.outlier_p
    vm = torch.rand(shape, generator=gen, device=device) < wl.outlier_p
    k = torch.where(km, k * wl.outlier_factor, k).to(torch.bfloat16)
    v = torch.where(vm, v * wl.outlier_factor, v).to(torch.bfloat16)
    rng = np.random.default_rng(wl.seed)
    slots = rng.permutation(wl.num_blocks * wl.block_size)[:wl.N].astype(np.int64)
    return k, v, torch.from_numpy(slots).to(device)


def dequant_workload(name: str = "dequant") -> DecodeWorkload:
    """One long sequence whose cached prefix is expanded to bf16.

    dequant        L=32768 (2048 pages), Hk=8 (Hq=64, unused by the kernel), seed 6
    dequant_small  L=1000 (63 pages, ragged last page), Hk=3, seed 7
    """
    if name == "dequant":
        return make_decode_workload("dequant", 1, 64, 8, np.array([32768]), 32768 // BLOCK_SIZE, 1,
                                    seed=6, spare_blocks=5)
    if name == "dequant_small":
        return make_decode_workload("dequant_small", 1, 18, 3, np.array([1000]), 64, 1, seed=7,
                                    spare_blocks=2)
    raise KeyError(name)


def dequant_bytes(wl: DecodeWorkload) -> int:
    """Bytes one full dequantisation moves: whole pages read (272 B per
    (token, kv head)), bf16 K and V written (1024 B), page ids read."""
    pages = int((int(wl.seq_lens[0]) + wl.block_size - 1) // wl.block_size)
    rows = pages * wl.block_size * wl.Hk
    return rows * (wl.D + wl.D // 16) + rows * wl.D * 2 * 2 + pages * 4


def multi_query_workload(name: str = "mq"):
    """A continuation chunk of q_len tokens after cached_len cached tokens of
    one sequence (all cached_len + q_len tokens stored); returns (wl, cached_len, q_len).

    mq   cached 131072 + 8 draft tokens, Hq=64, Hk=8 (GQA 8), S=32, seed 8
    """
    if name == "mq":
        cached, q_len = 131072, 8
        L = cached + q_len
        wl = make_decode_workload("mq", 1, 64, 8, np.array([L]), (L + BLOCK_SIZE - 1) // BLOCK_SIZE, 32,
                                  seed=8)
        return wl, cached, q_len
    raise KeyError(name)
