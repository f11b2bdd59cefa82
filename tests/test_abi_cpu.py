"""CPU-only checks of the C ABI: the library loads, exports every symbol that
include/uq.h declares, and rejects invalid arguments on the host before any
CUDA call (so these run without a GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from bit_quantized_kv_gb300 import binding
from bit_quantized_kv_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "uq.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(uq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert set(_declared_functions()) == set(binding.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_sizes_and_version(lib):
    assert lib.uq_version() >= 100
    assert lib.uq_slot_bytes(256) == 272
    assert lib.uq_slot_bytes(128) == 0
    n = lib.uq_decode_workspace_bytes(64, 48, 256, 32)
    assert n == ((64 * 48 * 32 * 1032 + 12 * 64 + 64 + 255) // 256) * 256
    assert lib.uq_decode_workspace_bytes(1, 8, 128, 4) == 0
    assert lib.uq_decode_workspace_bytes(1, 8, 256, 0) == 0
    assert lib.uq_decode_workspace_bytes(1, 8, 256, 257) == 0
    assert lib.uq_decode_workspace_bytes(0, 8, 256, 4) == 0


FAKE = 0x10000  # aligned, never dereferenced: validation returns first


def _decode(lib, **kw):
    args = dict(query=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, scale=0.0625, S=4, ws=FAKE,
                ws_bytes=1 << 30, out=FAKE, B=1, Hq=8, Hk=1, D=256, nb=32, bs=16, mb=32,
                sb=272, qss=8 * 256, qsh=256)
    args.update(kw)
    return lib.uq_decode(args["query"], args["kv"], args["bt"], args["sl"], args["scale"],
                         args["S"], args["ws"], args["ws_bytes"], args["out"], args["B"],
                         args["Hq"], args["Hk"], args["D"], args["nb"], args["bs"], args["mb"],
                         args["sb"], args["qss"], args["qsh"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=128), binding.UQ_ERR_UNSUPPORTED),
    (dict(bs=24), binding.UQ_ERR_UNSUPPORTED),
    (dict(bs=512), binding.UQ_ERR_UNSUPPORTED),
    (dict(Hq=4), binding.UQ_ERR_UNSUPPORTED),            # GQA 4
    (dict(Hq=12, Hk=1, qss=12 * 256), binding.UQ_ERR_UNSUPPORTED),
    (dict(Hq=9, Hk=2), binding.UQ_ERR_INVALID_ARG),      # not a multiple
    (dict(sb=288), binding.UQ_ERR_INVALID_ARG),
    (dict(S=0), binding.UQ_ERR_INVALID_ARG),
    (dict(S=257), binding.UQ_ERR_INVALID_ARG),
    (dict(query=0), binding.UQ_ERR_INVALID_ARG),
    (dict(out=0), binding.UQ_ERR_INVALID_ARG),
    (dict(ws=0), binding.UQ_ERR_INVALID_ARG),
    (dict(query=FAKE + 8), binding.UQ_ERR_INVALID_ARG),  # misaligned
    (dict(kv=FAKE + 4), binding.UQ_ERR_INVALID_ARG),
    (dict(qsh=200), binding.UQ_ERR_INVALID_ARG),
    (dict(qss=1000), binding.UQ_ERR_INVALID_ARG),
    (dict(nb=0), binding.UQ_ERR_INVALID_ARG),
    (dict(B=-1), binding.UQ_ERR_INVALID_ARG),
    (dict(B=70000), binding.UQ_ERR_INVALID_ARG),
    (dict(Hq=512 * 8, Hk=512, qss=512 * 8 * 256), binding.UQ_ERR_UNSUPPORTED),   # Hk > 256
    (dict(ws_bytes=1000), binding.UQ_ERR_WORKSPACE_TOO_SMALL),
    (dict(scale=float("nan")), binding.UQ_ERR_INVALID_ARG),
])
def test_decode_rejects_invalid_arguments(lib, kw, status):
    assert _decode(lib, **kw) == status
    assert lib.uq_last_error().decode() != ""


def test_decode_empty_batch_is_a_noop(lib):
    assert _decode(lib, B=0, query=0, out=0) == binding.UQ_OK
    assert lib.uq_last_error().decode() == ""


def _store(lib, **kw):
    args = dict(k=FAKE, v=FAKE, kv=FAKE, sm=FAKE, N=10, Hk=2, D=256, nb=4, bs=16, sb=272,
                ks=512, vs=512)
    args.update(kw)
    return lib.uq_store(args["k"], args["v"], args["kv"], args["sm"], args["N"], args["Hk"],
                        args["D"], args["nb"], args["bs"], args["sb"], args["ks"], args["vs"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=128), binding.UQ_ERR_UNSUPPORTED),
    (dict(sb=256), binding.UQ_ERR_INVALID_ARG),
    (dict(Hk=0), binding.UQ_ERR_INVALID_ARG),
    (dict(N=-1), binding.UQ_ERR_INVALID_ARG),
    (dict(k=0), binding.UQ_ERR_INVALID_ARG),
    (dict(sm=0), binding.UQ_ERR_INVALID_ARG),
    (dict(k=FAKE + 2), binding.UQ_ERR_INVALID_ARG),
    (dict(sm=FAKE + 4), binding.UQ_ERR_INVALID_ARG),
    (dict(ks=500), binding.UQ_ERR_INVALID_ARG),           # < Hk * D
    (dict(vs=516), binding.UQ_ERR_INVALID_ARG),           # not a multiple of 8
    (dict(nb=0), binding.UQ_ERR_INVALID_ARG),
])
def test_store_rejects_invalid_arguments(lib, kw, status):
    assert _store(lib, **kw) == status


def test_store_zero_tokens_is_a_noop(lib):
    assert _store(lib, N=0, k=0, v=0, kv=0, sm=0) == binding.UQ_OK


def test_store_rotated_rejects_invalid_arguments(lib):
    st = lib.uq_store_rotated_f32(FAKE, FAKE, FAKE, FAKE, 4, 1, 64, 1, 16, 272, None)
    assert st == binding.UQ_ERR_UNSUPPORTED
    st = lib.uq_store_rotated_f32(FAKE + 4, FAKE, FAKE, FAKE, 4, 1, 256, 1, 16, 272, None)
    assert st == binding.UQ_ERR_INVALID_ARG


def _mq(lib, **kw):
    args = dict(q=FAKE, kv=FAKE, bt=FAKE, cached=100, q_len=4, scale=0.0625, S=8, ws=FAKE,
                ws_bytes=1 << 30, out=FAKE, Hq=16, Hk=2, D=256, nb=64, bs=16, mb=8, sb=272,
                qst=16 * 256, qsh=256)
    args.update(kw)
    return lib.uq_decode_multi_query(args["q"], args["kv"], args["bt"], args["cached"], args["q_len"],
                                     args["scale"], args.get("sinks"), args.get("window", 0), args["S"],
                                     args["ws"], args["ws_bytes"], args["out"],
                                     args["Hq"], args["Hk"], args["D"], args["nb"], args["bs"], args["mb"],
                                     args["sb"], args["qst"], args["qsh"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(cached=-1), binding.UQ_ERR_INVALID_ARG),
    (dict(cached=126, q_len=3), binding.UQ_ERR_INVALID_ARG),   # 129 tokens > 8 pages
    (dict(q_len=-1), binding.UQ_ERR_INVALID_ARG),
    (dict(Hq=20), binding.UQ_ERR_UNSUPPORTED),                 # GQA 10
    (dict(ws_bytes=100), binding.UQ_ERR_WORKSPACE_TOO_SMALL),
    (dict(q=FAKE + 8), binding.UQ_ERR_INVALID_ARG),
    (dict(bt=0), binding.UQ_ERR_INVALID_ARG),
    (dict(sinks=FAKE + 2), binding.UQ_ERR_INVALID_ARG),
])
def test_multi_query_rejects_invalid_arguments(lib, kw, status):
    assert _mq(lib, **kw) == status
    assert lib.uq_last_error().decode() != ""


def test_multi_query_empty_chunk_is_a_noop(lib):
    assert _mq(lib, q_len=0, q=0, out=0, ws=0) == binding.UQ_OK


def _dequant(lib, **kw):
    args = dict(kv=FAKE, bt=FAKE, n=3, k=FAKE, v=FAKE, Hk=2, D=256, nb=4, bs=16, sb=272)
    args.update(kw)
    return lib.uq_full_dequant(args["kv"], args["bt"], args["n"], args["k"], args["v"], args["Hk"],
                               args["D"], args["nb"], args["bs"], args["sb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=128), binding.UQ_ERR_UNSUPPORTED),
    (dict(bs=48), binding.UQ_ERR_UNSUPPORTED),
    (dict(Hk=0), binding.UQ_ERR_UNSUPPORTED),
    (dict(Hk=300), binding.UQ_ERR_UNSUPPORTED),
    (dict(sb=288), binding.UQ_ERR_INVALID_ARG),
    (dict(nb=0), binding.UQ_ERR_INVALID_ARG),
    (dict(n=-1), binding.UQ_ERR_INVALID_ARG),
    (dict(n=1 << 27), binding.UQ_ERR_INVALID_ARG),         # n * 16 >= 2^31
    (dict(n=1 << 24, Hk=256), binding.UQ_ERR_INVALID_ARG), # n * Hk >= 2^31
    (dict(kv=0), binding.UQ_ERR_INVALID_ARG),
    (dict(k=0), binding.UQ_ERR_INVALID_ARG),
    (dict(k=FAKE + 8), binding.UQ_ERR_INVALID_ARG),        # misaligned
    (dict(bt=FAKE + 2), binding.UQ_ERR_INVALID_ARG),
])
def test_full_dequant_rejects_invalid_arguments(lib, kw, status):
    assert _dequant(lib, **kw) == status
    assert lib.uq_last_error().decode() != ""


def test_full_dequant_zero_pages_is_a_noop(lib):
    assert _dequant(lib, n=0, kv=0, bt=0, k=0, v=0) == binding.UQ_OK


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 8, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.uq_decode(q, torch.zeros(1, 16, 1, 272, dtype=torch.uint8),
                          torch.zeros(1, 1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32),
                          0.0625, 4, torch.zeros(16, dtype=torch.uint8), q.clone())


def test_python_binding_checks_dtypes_and_devices(lib):
    """The torch-facing wrappers reject wrong dtypes, ranks and host tensors
    before any call into the library."""
    import torch
    cache = torch.zeros(2, 16, 1, 272, dtype=torch.uint8)
    q = torch.zeros(3, 8, 256, dtype=torch.bfloat16)
    bt = torch.zeros(2, dtype=torch.int32)
    ws = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(ValueError):           # host tensors
        binding.uq_decode_multi_query(q, cache, bt, 10, 0.0625, 4, ws, q.clone())
    with pytest.raises(TypeError):            # fp32 query
        binding.uq_decode_multi_query(q.float(), cache, bt, 10, 0.0625, 4, ws, q.clone())
    with pytest.raises(ValueError):           # 2-D block table for one sequence
        binding.uq_decode_multi_query(q, cache, bt.view(1, 2), 10, 0.0625, 4, ws, q.clone())
    k = torch.zeros(1, 32, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.uq_full_dequant(cache, bt, k, k.clone())
    with pytest.raises(TypeError):            # int8 cache (checked first)
        binding.uq_full_dequant(cache.to(torch.int8), bt, k, k.clone())


@pytest.mark.parametrize("wrapper", ["uq_decode", "uq_decode_ex", "uq_decode_static_scratch"])
def test_batch_decode_wrappers_check_table_layout_before_the_device(lib, wrapper):
    """Every batch decode wrapper refuses a column slice of the block table
    (its row stride would be passed as the width) and a block table or
    seq_lens with fewer rows than the batch (the kernels would read past
    them), before anything reaches the library or the GPU."""
    import torch
    B = 4
    q = torch.zeros(B, 8, 256, dtype=torch.bfloat16)
    cache = torch.zeros(8, 16, 1, 272, dtype=torch.uint8)
    ws = torch.zeros(64, dtype=torch.uint8)

    def call(bt, sl):
        if wrapper == "uq_decode":
            binding.uq_decode(q, cache, bt, sl, 0.0625, 4, ws, q.clone())
        elif wrapper == "uq_decode_ex":
            binding.uq_decode_ex(q, cache, bt, sl, 0.0625, None, 0, 4, ws, q.clone())
        else:
            binding.uq_decode_static_scratch(q, cache, bt, sl, 0.0625, 4, q.clone())

    wide = torch.zeros(B, 6, dtype=torch.int32)
    lens = torch.zeros(B, dtype=torch.int32)
    with pytest.raises(ValueError, match="contiguous"):
        call(wide[:, 1:4], lens)                 # a column slice: row stride 6, width 3
    with pytest.raises(ValueError, match="fewer rows"):
        call(wide, lens[:B - 1])                 # seq_lens shorter than the batch
    with pytest.raises(ValueError, match="fewer rows"):
        call(wide[:B - 2], lens)                 # block table shorter than the batch
    with pytest.raises(ValueError, match="CUDA"):
        call(wide, lens)                         # well formed, but host tensors
