"""Helpers shared by the GPU parity tests: build caches through the CUDA
library and through the oracle from the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_quantized_kv_gb300 import binding, workloads
from bit_quantized_kv_gb300.build import build

# Decode tolerance: bf16 output against the fp64 oracle on the same packed
# cache (max-abs and relative L2 over the compared elements).
MAX_ABS = 1e-2
REL_L2 = 5e-3


def lib():
    build()
    return binding.load()


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def compare(gpu_bf16: torch.Tensor, ref: np.ndarray, max_abs=MAX_ABS, rel_l2=REL_L2):
    got = gpu_bf16.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(got).all(), "non-finite GPU output"
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    den = float(np.linalg.norm(ref))
    rl2 = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))
    assert mx <= max_abs, f"max-abs error {mx:.3e} > {max_abs}"
    assert rl2 <= rel_l2, f"relative L2 error {rl2:.3e} > {rel_l2}"
    return mx, rl2


def fill_cache_gpu(wl: workloads.DecodeWorkload, device="cuda") -> torch.Tensor:
    """Store every sequence of `wl` into a fresh cache with uq_store."""
    cache = torch.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), dtype=torch.uint8, device=device)
    for b in range(wl.B):
        if wl.seq_lens[b] == 0:
            continue
        k, v = workloads.sequence_kv(wl, b, device)
        slots = torch.from_numpy(workloads.sequence_slots(wl, b)).to(device)
        binding.uq_store(k, v, cache, slots)
    return cache


def oracle_cache_for_sequence(wl: workloads.DecodeWorkload, b: int, device="cuda"):
    """The oracle's own packed pages of sequence b (compact: page i of the
    sequence at cache page i), built from the same seeded bf16 inputs."""
    k, v = workloads.sequence_kv(wl, b, device)
    L = int(wl.seq_lens[b])
    P = (L + wl.block_size - 1) // wl.block_size
    cache = np.zeros((max(P, 1), wl.block_size, wl.Hk, 272), np.uint8)
    oracle.store(bits(k), bits(v), np.arange(L, dtype=np.int64), cache)
    return cache


def gpu_pages_of_sequence(cache: torch.Tensor, wl: workloads.DecodeWorkload, b: int) -> np.ndarray:
    L = int(wl.seq_lens[b])
    P = (L + wl.block_size - 1) // wl.block_size
    idx = torch.as_tensor(wl.block_table[b, :P].astype(np.int64), device=cache.device)
    return cache.index_select(0, idx).cpu().numpy()


def run_decode(wl: workloads.DecodeWorkload, cache: torch.Tensor, q: torch.Tensor,
               splits: int | None = None, seq_lens=None, block_table=None) -> torch.Tensor:
    dev = cache.device
    S = wl.splits if splits is None else splits
    bt = torch.from_numpy(wl.block_table if block_table is None else block_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens if seq_lens is None else seq_lens).to(dev)
    ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, wl.D, S), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device=dev)
    binding.uq_decode(q, cache, bt, sl, wl.scale, S, ws, out)
    return out


def oracle_rows(wl: workloads.DecodeWorkload, q: torch.Tensor, rows, device="cuda") -> np.ndarray:
    """Oracle output rows [(b, r), ...], each from the oracle's own cache of
    sequence b; also checks that those cache pages match the GPU's bytes."""
    qb = bits(q)
    out = []
    per_seq = {}
    for b, r in rows:
        if b not in per_seq:
            per_seq[b] = oracle_cache_for_sequence(wl, b, device)
        c = per_seq[b]
        L = int(wl.seq_lens[b])
        P = c.shape[0]
        bt = np.arange(P, dtype=np.int32)[None]
        o = oracle.decode(qb[b:b + 1], c, bt, np.array([L], np.int32), wl.scale,
                          rows=np.array([[0, r]], np.int32))
        out.append(o[0])
    return np.stack(out), per_seq
