"""CPU oracle for the UltraQuant 4-bit KV cache (test infrastructure).

This package is test infrastructure: only ``tests/``, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` import it.  It wraps the plain C,
fp64 implementation in ``uq_oracle.c`` through ctypes and shares no code with
the CUDA library in ``bit_quantized_kv_gb300``.

Functions take and return numpy arrays.  bf16 tensors are passed as their
uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle

_LIB = None


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    global _LIB
    if _LIB is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        c_int, c_i64, c_dbl, c_p = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.uqo_bf16_to_double.restype = c_dbl
        L.uqo_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.uqo_round_format.restype = c_dbl
        L.uqo_round_format.argtypes = [c_dbl, c_int, c_int, c_dbl, c_int]
        L.uqo_bf16_round.restype = ctypes.c_uint16
        L.uqo_bf16_round.argtypes = [c_dbl]
        L.uqo_e4m3_round.restype = c_dbl
        L.uqo_e4m3_round.argtypes = [c_dbl]
        L.uqo_e2m1_value.restype = c_dbl
        L.uqo_e2m1_value.argtypes = [c_int]
        L.uqo_e2m1_encode.restype = c_int
        L.uqo_e2m1_encode.argtypes = [c_dbl]
        L.uqo_ue8m0_byte.restype = c_int
        L.uqo_ue8m0_byte.argtypes = [c_dbl]
        L.uqo_hadamard.restype = None
        L.uqo_hadamard.argtypes = [c_int, c_p]
        L.uqo_fwht_f32.restype = None
        L.uqo_fwht_f32.argtypes = [c_p, c_int]
        L.uqo_slot_bytes.restype = c_int
        L.uqo_slot_bytes.argtypes = [c_int]
        L.uqo_quantize_slot.restype = None
        L.uqo_quantize_slot.argtypes = [c_p, c_p, c_int, c_p]
        L.uqo_dequant_slot.restype = None
        L.uqo_dequant_slot.argtypes = [c_p, c_int, c_p, c_p]
        L.uqo_store.restype = c_i64
        L.uqo_store.argtypes = [c_p, c_p, c_p, c_i64, c_int, c_int, c_i64, c_i64,
                                c_int, c_int, c_p]
        L.uqo_store_f32.restype = c_i64
        L.uqo_store_f32.argtypes = [c_p, c_p, c_p, c_i64, c_int, c_int, c_int, c_int, c_p]
        L.uqo_decode_ex.restype = c_int
        L.uqo_decode_ex.argtypes = [c_p, c_i64, c_i64, c_p, c_p, c_p, c_dbl,
                                    c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                    c_p, c_int, c_p, c_int, c_int, c_p]
        L.uqo_full_dequant.restype = c_int
        L.uqo_full_dequant.argtypes = [c_p, c_p, c_int, c_int, c_int, c_int, c_int, c_p, c_p]
        L.uqo_query_prime.restype = None
        L.uqo_query_prime.argtypes = [c_p, c_int, c_p, c_p]
        L.uqo_decode.restype = c_int
        L.uqo_decode.argtypes = [c_p, c_i64, c_i64, c_p, c_p, c_p, c_dbl,
                                 c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                 c_p, c_int, c_int, c_p]
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


# --------------------------------------------------------------------------- #
# Scalar format helpers                                                        #
# --------------------------------------------------------------------------- #

def round_format(x: float, mant_bits: int, emin: int, maxval: float, satfinite: bool) -> float:
    return lib().uqo_round_format(float(x), mant_bits, emin, float(maxval), int(satfinite))


def e2m1_value(code: int) -> float:
    return lib().uqo_e2m1_value(int(code))


def e2m1_encode(y: float) -> int:
    return lib().uqo_e2m1_encode(float(y))


def ue8m0_byte(amax: float) -> int:
    return lib().uqo_ue8m0_byte(float(amax))


def e4m3_round(x: float) -> float:
    return lib().uqo_e4m3_round(float(x))


def bf16_round(x: float) -> int:
    return lib().uqo_bf16_round(float(x))


def bf16_round_array(x: np.ndarray) -> np.ndarray:
    """Round an fp64 array to bf16 bit patterns (round to nearest even)."""
    f = lib().uqo_bf16_round
    flat = np.ascontiguousarray(x, dtype=np.float64).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(x))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 bit pattern -> float64 conversion."""
    u = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- #
# Rotation and packing                                                         #
# --------------------------------------------------------------------------- #

def hadamard(D: int) -> np.ndarray:
    H = np.empty((D, D), dtype=np.float64)
    lib().uqo_hadamard(D, _ptr(H))
    return H


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """Canonical-order unnormalised fp32 FWHT of a 1-D array."""
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    lib().uqo_fwht_f32(_ptr(y), y.shape[0])
    return y


def slot_bytes(D: int = 256) -> int:
    return lib().uqo_slot_bytes(D)


def quantize_slot(k_rot: np.ndarray, v: np.ndarray) -> np.ndarray:
    k_rot = np.ascontiguousarray(k_rot, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    D = k_rot.shape[0]
    out = np.zeros(slot_bytes(D), dtype=np.uint8)
    lib().uqo_quantize_slot(_ptr(k_rot), _ptr(v), D, _ptr(out))
    return out


def dequant_slot(slot: np.ndarray, D: int = 256):
    slot = np.ascontiguousarray(slot, dtype=np.uint8)
    k = np.empty(D, dtype=np.float64)
    v = np.empty(D, dtype=np.float64)
    lib().uqo_dequant_slot(_ptr(slot), D, _ptr(k), _ptr(v))
    return k, v


def store(key_bits: np.ndarray, value_bits: np.ndarray, slot_mapping: np.ndarray,
          kv_cache: np.ndarray) -> int:
    """Quantise bf16 K [N,Hk,D] (rotated here) and V into ``kv_cache`` in place.

    ``kv_cache`` is uint8 [num_blocks, block_size, Hk, slot].  Returns the
    number of skipped (negative-slot) rows, or -1 for a slot beyond the cache.
    """
    key_bits = np.ascontiguousarray(key_bits, dtype=np.uint16)
    value_bits = np.ascontiguousarray(value_bits, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    N, Hk, D = key_bits.shape
    nb, bs, hk2, sbytes = kv_cache.shape
    assert hk2 == Hk and sbytes == slot_bytes(D) and kv_cache.flags["C_CONTIGUOUS"]
    return lib().uqo_store(_ptr(key_bits), _ptr(value_bits), _ptr(sm), N, Hk, D,
                           Hk * D, Hk * D, nb, bs, _ptr(kv_cache))


def store_f32(k_rot: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray,
              kv_cache: np.ndarray) -> int:
    """Quantise pre-rotated fp32 K [N,Hk,D] and fp32 V into ``kv_cache``."""
    k_rot = np.ascontiguousarray(k_rot, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    N, Hk, D = k_rot.shape
    nb, bs, _, _ = kv_cache.shape
    return lib().uqo_store_f32(_ptr(k_rot), _ptr(v), _ptr(sm), N, Hk, D, nb, bs,
                               _ptr(kv_cache))


def full_dequant(kv_cache: np.ndarray, block_table: np.ndarray, n_pages: int | None = None):
    """Dequantise one sequence's pages into bf16 bit patterns.

    kv_cache: uint8 [num_blocks, block_size, Hk, slot]; block_table: int32
    page ids of the sequence.  Returns (k_bits, v_bits, n_bad_pages) with
    k_bits, v_bits uint16 [Hk, n_pages * block_size, D] (K still rotated).
    """
    bt = np.ascontiguousarray(block_table, dtype=np.int32).reshape(-1)
    n = int(bt.shape[0]) if n_pages is None else int(n_pages)
    kv_cache = np.ascontiguousarray(kv_cache, dtype=np.uint8)
    nb, bs, Hk, sbytes = kv_cache.shape
    D = (sbytes // 17) * 16
    assert sbytes == slot_bytes(D)
    k = np.zeros((Hk, n * bs, D), dtype=np.uint16)
    v = np.zeros((Hk, n * bs, D), dtype=np.uint16)
    bad = lib().uqo_full_dequant(_ptr(kv_cache), _ptr(bt), n, Hk, D, nb, bs, _ptr(k), _ptr(v))
    return k, v, int(bad)


def query_prime(q_bits: np.ndarray) -> np.ndarray:
    """Rotated, E4M3-rounded query row q' (fp64 values) of one bf16 row."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    D = q_bits.shape[0]
    H = hadamard(D)
    out = np.empty(D, dtype=np.float64)
    lib().uqo_query_prime(_ptr(q_bits), D, _ptr(H), _ptr(out))
    return out


def decode(query_bits: np.ndarray, kv_cache: np.ndarray, block_table: np.ndarray,
           seq_lens: np.ndarray, scale: float, splits: int = 0,
           rows: np.ndarray | None = None, nthreads: int | None = None,
           sinks: np.ndarray | None = None, window: int = 0) -> np.ndarray:
    """fp64 decode attention.

    query_bits: uint16 [B, Hq, D]; kv_cache: uint8 [nb, bs, Hk, slot];
    block_table: int32 [B, max_blocks]; seq_lens: int32 [B].  Optional sink
    logits [Hq] and a sliding window (> 0: the last ``window`` tokens).
    Returns fp64 [B, Hq, D], or [len(rows), D] when ``rows`` (an int32 [n, 2]
    array of (b, r) pairs) is given.
    """
    q = np.ascontiguousarray(query_bits, dtype=np.uint16)
    kv = np.ascontiguousarray(kv_cache, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    nb, bs, Hk, _ = kv.shape
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    if rows is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rows_p, n_rows = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((rows.shape[0], D), dtype=np.float64)
        rows_p, n_rows = _ptr(rows), rows.shape[0]
    sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64).reshape(Hq)
    rc = lib().uqo_decode_ex(_ptr(q), Hq * D, D, _ptr(kv), _ptr(bt), _ptr(sl), float(scale),
                             B, Hq, Hk, D, nb, bs, bt.shape[1], int(splits),
                             rows_p, n_rows, None if sk is None else _ptr(sk), int(window),
                             int(nthreads), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle decode failed ({rc})")
    return out
