#!/usr/bin/env python3
"""Benchmark of the FP4-KV decode step on GB300.

One step is the whole hot path for one decode step of a batch: uq_store of
each sequence's new token (K rotated and packed into the last slot of the
sequence) followed by uq_decode (query prologue, split-KV stage 1, LSE merge
stage 2) over the paged FP4 cache.  Inputs are seeded synthetic tensors
(bit_quantized_kv_gb300.workloads); the packed cache is built once, untimed,
with uq_store.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl uq|reference]

Prints ONE JSON line on rank 0.  ``value`` is achieved HBM GB/s of the whole
step (algorithmic bytes: packed KV read + bf16 query read + bf16 output
written + the store's bytes, divided by the device time of a step), summed
over ranks.  Under torchrun every rank runs its own copy of the workload
(weak scaling; no collective on the data path; gloo carries only the
barrier and the max-over-ranks timing).

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload on the host cores (the pages ship no runnable reference).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP4-KV decode attn: achieved HBM GB/s (% of peak), decode tokens/s"
DEFAULT_WORKLOAD = "outlier_long"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["bit_quantized_kv_gb300/csrc/uq_decode.cu", "bit_quantized_kv_gb300/csrc/uq_decode_common.cuh",
                  "bit_quantized_kv_gb300/csrc/uq_device.cuh"]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


DEQUANT_SOURCES = ["bit_quantized_kv_gb300/csrc/uq_dequant.cu", "bit_quantized_kv_gb300/csrc/uq_device.cuh"]
STORE_SOURCES = ["bit_quantized_kv_gb300/csrc/uq_store.cu", "bit_quantized_kv_gb300/csrc/uq_device.cuh"]


def _code_only(text: str) -> str:
    """C/C++ source with its comments and blank lines removed, so that a
    comment-only edit does not count as a changed kernel.  String literals
    are kept as they are (the sources' strings are PTX, which holds no
    comment markers)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def _source_hash(sources=None) -> str:
    """Hash of the code (comments stripped) of the files a profile covers."""
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic_from_profile(workload: str, profile: str | None = None, sources=None):
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu summary, if it was taken on the current kernel source; else
    None."""
    path = os.path.join(ROOT, "profiles", profile or f"decode_stage1_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, _, v = line.strip()[2:].partition(":")
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != _source_hash(sources):
        return None
    for key in ("dram_bytes_per_launch_full_size", "dram_bytes_per_launch"):
        try:
            return float(vals[key])
        except (KeyError, ValueError):
            continue
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def _dist_init():
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return rank, local, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(name: str, rank: int, world: int):
    """Weak scaling: every rank runs the same shape with its own seed, so the
    ranks' (sequence, kv head) units are independent replicas of the workload."""
    from bit_quantized_kv_gb300 import workloads
    wl = workloads.decode_workload(name)
    if world > 1:
        wl.seed = wl.seed + 1000 * rank
    return wl


# --------------------------------------------------------------------------- #
# GPU arm                                                                      #
# --------------------------------------------------------------------------- #

class DecodeStep:
    """Device-resident state of one decode workload and its step."""

    def __init__(self, wl, device):
        import torch
        from bit_quantized_kv_gb300 import binding, workloads
        self.torch, self.binding, self.wl = torch, binding, wl
        self.dev = device
        t0 = time.time()
        self.cache = torch.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), dtype=torch.uint8, device=device)
        for b in range(wl.B):
            if wl.seq_lens[b] == 0:
                continue
            k, v = workloads.sequence_kv(wl, b, device)
            slots = torch.from_numpy(workloads.sequence_slots(wl, b)).to(device)
            binding.uq_store(k, v, self.cache, slots)
            del k, v
        torch.cuda.synchronize()
        self.fill_s = time.time() - t0
        self.q = workloads.query(wl, device)
        self.k_new, self.v_new = workloads.new_token_kv(wl, device)
        self.slots_new = torch.from_numpy(workloads.last_slots(wl)).to(device)
        self.bt = torch.from_numpy(wl.block_table).to(device)
        self.sl = torch.from_numpy(wl.seq_lens).to(device)
        self.ws = torch.empty(binding.uq_decode_workspace_bytes(wl.B, wl.Hq, wl.D, wl.splits),
                              dtype=torch.uint8, device=device)
        self.out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device=device)

    def step(self):
        b = self.binding
        b.uq_store(self.k_new, self.v_new, self.cache, self.slots_new)
        b.uq_decode(self.q, self.cache, self.bt, self.sl, self.wl.scale, self.wl.splits, self.ws, self.out)

    def store_bytes(self) -> int:
        wl = self.wl
        return wl.B * wl.Hk * (2 * wl.D * 2 + 272) + 8 * wl.B

    def bytes_per_step(self) -> int:
        return self.wl.algorithmic_bytes() + self.store_bytes()


def run_gpu(args, rank, local, world):
    import torch
    from bit_quantized_kv_gb300 import binding
    from bit_quantized_kv_gb300.build import build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    binding.load()
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = _peaks()

    if args.workload == "store":
        return run_gpu_store(args, rank, local, world, dev, stream, peak, peak_kind)
    if args.workload == "dequant":
        return run_gpu_dequant(args, rank, local, world, dev, stream, peak, peak_kind)
    if args.workload == "mq":
        return run_gpu_mq(args, rank, local, world, dev, stream, peak, peak_kind)

    wl = rank_workload(args.workload, rank, world)
    line, st = measure_decode(args, wl, dev, stream, peak, peak_kind, local, world)
    with torch.cuda.stream(stream):
        # end to end through the public API: pinned host inputs in, output back out
        line["e2e"] = run_e2e(args, st, stream, torch)
    del st
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args)
    if args.workload == DEFAULT_WORKLOAD and not args.headline_only:
        line["workloads"] = other_workloads(args, rank, local, world, dev, stream, peak, peak_kind)
    return line


def measure_decode(args, wl, dev, stream, peak, peak_kind, local, world):
    """Time `args.steps` decode steps (store of the B new tokens + decode) of a
    decode workload after `args.warmup` untimed ones, with stage 1 timed alone
    on its stream; return (JSON fields, the DecodeStep)."""
    import torch
    from bit_quantized_kv_gb300 import binding
    with torch.cuda.stream(stream):
        st = DecodeStep(wl, dev)
        torch.cuda.synchronize()
        use_graph = wl.graph_replay
        graph = None
        if use_graph:
            st.step()  # eager warm-up before capture
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                st.step()
        run = graph.replay if use_graph else st.step
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()

        n = args.steps
        # pass 1: the timed steps, with no event between the kernels (so each
        # kernel may start while the one before it finishes)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        _barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(local) as clocks:
            start.record(stream)
            for _ in range(n):
                run()
            end.record(stream)
            torch.cuda.synchronize()
        _barrier(world)
        torch.cuda.synchronize()
        total_ms = start.elapsed_time(end)

        # pass 2: the same steps with stage 1 bracketed by events on the
        # launching stream, for the stage-1 roofline
        ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in ev_b + ev_a:
            e.record(stream)  # materialise the handles
        torch.cuda.synchronize()
        if use_graph:
            # re-capture with the timing events inside the graph: one graph per step
            graphs = []
            for i in range(n):
                binding.uq_set_timing_events(ev_b[i], ev_a[i])
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st.step()
                graphs.append(g)
            binding.uq_set_timing_events(None, None)
            for g in graphs[:1]:
                g.replay()
            torch.cuda.synchronize()
        for i in range(n):
            if use_graph:
                graphs[i].replay()
            else:
                binding.uq_set_timing_events(ev_b[i], ev_a[i])
                st.step()
        binding.uq_set_timing_events(None, None)
        torch.cuda.synchronize()
        stage1_ms = [ev_b[i].elapsed_time(ev_a[i]) for i in range(n)]
        flags = binding.uq_check_device_error(stream)
        if flags:
            raise RuntimeError(f"device error flags 0x{flags:x} during the benchmark")
        if use_graph:
            del graphs, graph

    total_ms = _max_over_ranks(total_ms, world)
    ms_per_step = total_ms / n
    bytes_step = st.bytes_per_step()
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9
    s1_ms = statistics.mean(stage1_ms)
    kv_bytes = wl.kv_bytes() + wl.B * wl.Hq * wl.D * 2   # stage 1 reads packed KV + query
    achieved = kv_bytes / (s1_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp4-e2m1 cache, f16 mma, f32 accumulate", "data": "synthetic",
        "pct_of_peak": round(100.0 * bytes_step / (ms_per_step * 1e-3) / 1e9 / peak, 2),
        "decode_tokens_per_s": round(world * wl.B / (ms_per_step * 1e-3), 1),
        "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hk": wl.Hk, "D": wl.D,
                   "block_size": wl.block_size, "max_num_kv_splits": wl.splits,
                   "seq_len_total": int(wl.seq_lens.sum()),
                   "seq_len_min": int(wl.seq_lens.min()), "seq_len_max": int(wl.seq_lens.max()),
                   "cuda_graph": bool(wl.graph_replay),
                   "bytes_per_step": bytes_step,
                   "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB per step)"
                         if bytes_step > 129e6 else "inputs smaller than L2 (not flushed)",
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "kernel": "decode_stage1", "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": _traffic_from_profile(wl.name),
                     "stage1_ms": round(s1_ms, 5), "stage1_bytes": kv_bytes},
        "gpu_launches": n * 5,   # per step: store, plan, stage 1, exact pass, stage 2
        "clocks": clocks.summary(),
    }
    return line, st


# Workloads timed after the headline in the default run, each in its own
# section of the JSON line: the other decode configurations, the store, the
# multi-query continuation chunk and the full-prefix dequantisation.
EXTRA_WORKLOADS = ("skewed", "batch", "tiny", "store", "mq", "dequant")
EXTRA_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "pct_of_peak", "decode_tokens_per_s",
              "config", "roofline", "clocks", "gpu_launches")


def other_workloads(args, rank, local, world, dev, stream, peak, peak_kind):
    import torch
    out = {}
    for name in EXTRA_WORKLOADS:
        if name == "store":
            line = run_gpu_store(args, rank, local, world, dev, stream, peak, peak_kind)
        elif name == "mq":
            line = run_gpu_mq(args, rank, local, world, dev, stream, peak, peak_kind, cpu=False)
        elif name == "dequant":
            line = run_gpu_dequant(args, rank, local, world, dev, stream, peak, peak_kind, cpu=False)
        else:
            line, st = measure_decode(args, rank_workload(name, rank, world), dev, stream, peak,
                                      peak_kind, local, world)
            del st
        out[name] = {k: line[k] for k in EXTRA_KEYS if k in line}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_e2e(args, st, stream, torch):
    """Same step through the public API with host buffers: H2D of the step's
    inputs (query, new K/V, slots, seq_lens) from pinned memory, the two
    library calls, D2H of the output; timed with events on the stream."""
    binding = st.binding
    q_h = st.q.cpu().pin_memory()
    k_h = st.k_new.cpu().pin_memory()
    v_h = st.v_new.cpu().pin_memory()
    s_h = st.slots_new.cpu().pin_memory()
    l_h = st.sl.cpu().pin_memory()
    out_h = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h, s_h, l_h))
    d2h = out_h.numel() * out_h.element_size()

    def one():
        st.q.copy_(q_h, non_blocking=True)
        st.k_new.copy_(k_h, non_blocking=True)
        st.v_new.copy_(v_h, non_blocking=True)
        st.slots_new.copy_(s_h, non_blocking=True)
        st.sl.copy_(l_h, non_blocking=True)
        st.step()
        out_h.copy_(st.out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    return {"value": round(st.bytes_per_step() / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_gpu_store(args, rank, local, world, dev, stream, peak, peak_kind):
    import torch
    from bit_quantized_kv_gb300 import binding, workloads
    wl = workloads.store_workload("store")
    with torch.cuda.stream(stream):
        k, v, slots = workloads.store_inputs(wl, dev)
        cache = torch.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            binding.uq_store(k, v, cache, slots)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        _barrier(world)
        with ClockSampler(local) as clocks:
            for a, b in evs:
                a.record(stream)
                binding.uq_store(k, v, cache, slots)
                b.record(stream)
            torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
    total = _max_over_ranks(sum(ms), world)
    ms_step = total / args.steps
    by = wl.algorithmic_bytes()
    ach = by / (statistics.mean(ms) * 1e-3) / 1e9
    return {"metric": METRIC, "value": round(world * by / (ms_step * 1e-3) / 1e9, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, fp32 rotate, fp4-e2m1 out", "data": "synthetic",
            "config": {"workload": "store", "N": wl.N, "Hk": wl.Hk, "num_blocks": wl.num_blocks,
                       "bytes_per_step": by, "l2": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "store", "achieved": round(ach, 2), "peak": peak,
                         "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                         "frac": round(ach / peak, 4),
                         "traffic": _traffic_from_profile("store", "store_kernel_store.md", STORE_SOURCES)},
            "gpu_launches": args.steps, "clocks": clocks.summary()}


def run_gpu_dequant(args, rank, local, world, dev, stream, peak, peak_kind, cpu=True):
    """Full-prefix dequantisation of one 32768-token sequence (8 kv heads):
    each step expands its 2048 pages to bf16 K and V (340 MB moved per step,
    above L2)."""
    import torch
    from bit_quantized_kv_gb300 import binding, workloads
    wl = workloads.dequant_workload("dequant")
    n = wl.block_table.shape[1]
    with torch.cuda.stream(stream):
        cache = torch.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), dtype=torch.uint8, device=dev)
        k, v = workloads.sequence_kv(wl, 0, dev)
        binding.uq_store(k, v, cache, torch.from_numpy(workloads.sequence_slots(wl, 0)).to(dev))
        bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).to(dev)
        k_out = torch.empty((wl.Hk, n * wl.block_size, wl.D), dtype=torch.bfloat16, device=dev)
        v_out = torch.empty_like(k_out)
        for _ in range(args.warmup):
            binding.uq_full_dequant(cache, bt, k_out, v_out)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        _barrier(world)
        with ClockSampler(local) as clocks:
            for a, b in evs:
                a.record(stream)
                binding.uq_full_dequant(cache, bt, k_out, v_out)
                b.record(stream)
            torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
    total = _max_over_ranks(sum(ms), world)
    ms_step = total / args.steps
    by = workloads.dequant_bytes(wl)
    ach = by / (statistics.mean(ms) * 1e-3) / 1e9
    line = {"metric": METRIC, "value": round(world * by / (ms_step * 1e-3) / 1e9, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp4-e2m1 cache in, bf16 out", "data": "synthetic",
            "config": {"workload": "dequant", "seq_len": int(wl.seq_lens[0]), "pages": n,
                       "Hk": wl.Hk, "D": wl.D, "bytes_per_step": by,
                       "l2": "inputs and outputs larger than L2 (340 MB per step)"},
            "roofline": {"bound": "hbm", "kernel": "full_dequant", "achieved": round(ach, 2),
                         "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                         "frac": round(ach / peak, 4),
                         "traffic": _traffic_from_profile("dequant", "full_dequant_dequant.md", DEQUANT_SOURCES)},
            "gpu_launches": args.steps, "clocks": clocks.summary()}
    if rank == 0 and cpu and not args.no_cpu_baseline:
        nbytes, secs, desc = _oracle_dequant_sample(wl, args.cpu_budget)
        line["cpu_baseline"] = {"value": round(nbytes / secs / 1e9, 6), "unit": UNIT, "cores": 1,
                                "kind": "oracle", "sample": desc}
    return line


def run_gpu_mq(args, rank, local, world, dev, stream, peak, peak_kind, cpu=True):
    """Multi-query continuation decode: 8 draft tokens after 131072 cached
    tokens of one sequence (GQA 8).  GB/s counts each cached byte once (the
    8 rows share the pages; repeats come from L2)."""
    import torch
    from bit_quantized_kv_gb300 import binding, workloads
    wl, cached, q_len = workloads.multi_query_workload("mq")
    S = wl.splits
    with torch.cuda.stream(stream):
        cache = torch.zeros((wl.num_blocks, wl.block_size, wl.Hk, 272), dtype=torch.uint8, device=dev)
        k, v = workloads.sequence_kv(wl, 0, dev)
        binding.uq_store(k, v, cache, torch.from_numpy(workloads.sequence_slots(wl, 0)).to(dev))
        q = workloads.chunk_query(wl, q_len, dev)
        bt = torch.from_numpy(np.ascontiguousarray(wl.block_table[0])).to(dev)
        ws = torch.empty(binding.uq_decode_workspace_bytes(q_len, wl.Hq, wl.D, S), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        for _ in range(args.warmup):
            binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        s1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in s1:
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize()
        _barrier(world)
        with ClockSampler(local) as clocks:
            for (a, b), (c, d) in zip(evs, s1):
                binding.uq_set_timing_events(c, d)
                a.record(stream)
                binding.uq_decode_multi_query(q, cache, bt, cached, wl.scale, S, ws, out)
                b.record(stream)
            torch.cuda.synchronize()
        binding.uq_set_timing_events(None, None)
        ms = [a.elapsed_time(b) for a, b in evs]
        ms1 = [c.elapsed_time(d) for c, d in s1]
    total = _max_over_ranks(sum(ms), world)
    ms_step = total / args.steps
    kv_bytes = (cached + q_len) * wl.Hk * 272
    by = kv_bytes + 2 * q_len * wl.Hq * wl.D * 2
    ach = by / (statistics.mean(ms1) * 1e-3) / 1e9
    return {"metric": METRIC, "value": round(world * by / (ms_step * 1e-3) / 1e9, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp4-e2m1 cache, f16 mma, f32 accumulate", "data": "synthetic",
            "decode_tokens_per_s": round(world * q_len / (ms_step * 1e-3), 1),
            "config": {"workload": "mq", "cached_len": cached, "q_len": q_len, "Hq": wl.Hq, "Hk": wl.Hk,
                       "D": wl.D, "max_num_kv_splits": S, "bytes_per_step": by,
                       "l2": "cache larger than L2 (285 MB per step)"},
            "roofline": {"bound": "hbm", "kernel": "decode_stage1", "achieved": round(ach, 2),
                         "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                         "frac": round(ach / peak, 4), "traffic": _traffic_from_profile("mq"),
                         "stage1_ms": round(statistics.mean(ms1), 5)},
            "gpu_launches": args.steps * 4, "clocks": clocks.summary(),
            **({} if (rank != 0 or not cpu or args.no_cpu_baseline) else {"cpu_baseline": _mq_cpu_baseline(args.cpu_budget)})}


def _oracle_mq_sample(budget_s: float):
    """Time the oracle's decode of the mq workload's synthetic batch, one
    (chunk row, query head) at a time over the host cores, until about
    budget_s seconds; return (bytes, seconds, threads, description).  Bytes
    count the cached pages once per chunk row, as the GPU line does per step."""
    import torch
    import oracle
    from bit_quantized_kv_gb300 import workloads
    wl, cached, q_len = workloads.multi_query_workload("mq")
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    k, v = workloads.sequence_kv(wl, 0, dev)
    kb = k.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = v.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    L = cached + q_len
    P = (L + 15) // 16
    cache = np.zeros((P, 16, wl.Hk, 272), np.uint8)
    oracle.store(kb, vb, np.arange(L, dtype=np.int64), cache)          # untimed set-up
    q = workloads.chunk_query(wl, q_len, dev)
    qb = q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    table = np.tile(np.arange(P, dtype=np.int32), (q_len, 1))
    lens = (cached + 1 + np.arange(q_len)).astype(np.int32)
    threads = min(os.cpu_count() or 1, wl.Hq)
    spent, rows_done = 0.0, 0
    for i in range(q_len):
        rows = np.array([[i, r] for r in range(wl.Hq)], np.int32)
        t0 = time.perf_counter()
        oracle.decode(qb, cache, table, lens, wl.scale, rows=rows, nthreads=threads)
        spent += time.perf_counter() - t0
        rows_done += 1
        if spent >= budget_s:
            break
    nbytes = rows_done * ((cached + q_len) * wl.Hk * 272 / q_len + 2 * wl.Hq * wl.D * 2)
    desc = (f"{rows_done} of {q_len} chunk rows (all {wl.Hq} query heads) of workload mq; "
            f"oracle packing untimed")
    return nbytes, spent, threads, desc


def _mq_cpu_baseline(budget_s: float):
    nbytes, secs, threads, desc = _oracle_mq_sample(budget_s)
    return {"value": round(nbytes / secs / 1e9, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle", "sample": desc}


def _oracle_dequant_sample(wl, budget_s: float):
    """Time the oracle's full dequantisation over pages of its own packing of
    the dequant workload, one call per 64 pages, until about budget_s seconds;
    return (bytes, seconds, description)."""
    import torch
    import oracle
    from bit_quantized_kv_gb300 import workloads
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    k, v = workloads.sequence_kv(wl, 0, dev)
    kb = k.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = v.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    L = int(wl.seq_lens[0])
    P = (L + 15) // 16
    cache = np.zeros((P, 16, wl.Hk, 272), np.uint8)
    oracle.store(kb, vb, np.arange(L, dtype=np.int64), cache)          # untimed set-up
    spent, pages = 0.0, 0
    while spent < budget_s and pages < P:
        chunk = np.arange(pages, min(P, pages + 64), dtype=np.int32)
        t0 = time.perf_counter()
        oracle.full_dequant(cache, chunk)
        spent += time.perf_counter() - t0
        pages += len(chunk)
    nbytes = pages * 16 * wl.Hk * (272 + 1024) + 4 * pages
    return nbytes, spent, f"{pages} of {P} pages of workload dequant (1 thread); oracle packing untimed"


# --------------------------------------------------------------------------- #
# CPU oracle (baseline / reference arm)                                        #
# --------------------------------------------------------------------------- #

def _oracle_sample(wl, budget_s: float):
    """Time the fp64 oracle's decode of whole sequences of the workload (every
    query head, rows spread over the host cores) until about budget_s seconds
    of CPU work; return (bytes processed, seconds, threads, description)."""
    import torch
    import oracle
    from bit_quantized_kv_gb300 import workloads
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    rng = np.random.default_rng(1234)
    order = rng.permutation(wl.B)
    q = workloads.query(wl, dev)
    qb = q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    threads = min(os.cpu_count() or 1, wl.Hq)
    done_bytes, spent, seqs, toks = 0, 0.0, 0, 0
    for b in order:
        L = int(wl.seq_lens[b])
        if L == 0:
            continue
        k, v = workloads.sequence_kv(wl, int(b), dev)
        kb = k.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        vb = v.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        P = (L + 15) // 16
        cache = np.zeros((P, 16, wl.Hk, 272), np.uint8)
        oracle.store(kb, vb, np.arange(L, dtype=np.int64), cache)      # untimed set-up
        t0 = time.perf_counter()
        oracle.decode(qb[b:b + 1], cache, np.arange(P, dtype=np.int32)[None],
                      wl.seq_lens[b:b + 1], wl.scale, nthreads=threads)
        spent += time.perf_counter() - t0
        done_bytes += L * wl.Hk * 272 + 2 * wl.Hq * wl.D * 2
        seqs += 1
        toks += L
        if spent >= budget_s:
            break
    desc = (f"{seqs} sequences ({toks} tokens, all {wl.Hq} query heads) of workload "
            f"{wl.name}; oracle decode only, its packing untimed")
    return done_bytes, spent, threads, desc


def cpu_baseline(wl, args):
    nbytes, secs, threads, desc = _oracle_sample(wl, args.cpu_budget)
    return {"value": round(nbytes / secs / 1e9, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle", "sample": desc}


def run_reference(args, rank, world):
    from bit_quantized_kv_gb300 import workloads
    if rank != 0:
        return None
    if args.workload == "dequant":
        return run_reference_dequant(args, world)
    if args.workload == "mq":
        per_step = max(1.0, args.cpu_budget / max(1, args.steps + args.warmup))
        tot_b, tot_s, desc, threads = 0.0, 0.0, "", 1
        for it in range(args.warmup + args.steps):
            b, sec, threads, desc = _oracle_mq_sample(per_step)
            if it >= args.warmup:
                tot_b += b
                tot_s += sec
        val = tot_b / tot_s / 1e9
        return {"metric": METRIC, "value": round(val, 6), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "impl": "reference", "config": {"workload": "mq"},
                "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": threads,
                                 "kind": "oracle", "sample": "each step: " + desc},
                "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
    wl = workloads.decode_workload(args.workload) if args.workload != "store" else None
    if wl is None:
        return {"impl": "reference", "unavailable": "store workload has no oracle timing arm"}
    per_step = max(1.0, args.cpu_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_sample(wl, per_step)
    tot_b, tot_s, desc, threads = 0, 0.0, "", 1
    for _ in range(args.steps):
        b, s, threads, desc = _oracle_sample(wl, per_step)
        tot_b += b
        tot_s += s
    val = tot_b / tot_s / 1e9
    return {"metric": METRIC, "value": round(val, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hk": wl.Hk, "D": wl.D},
            "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": "each step: " + desc},
            "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_reference_dequant(args, world):
    from bit_quantized_kv_gb300 import workloads
    wl = workloads.dequant_workload("dequant")
    per_step = max(1.0, args.cpu_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_dequant_sample(wl, per_step)
    tot_b, tot_s, desc = 0, 0.0, ""
    for _ in range(args.steps):
        b, sec, desc = _oracle_dequant_sample(wl, per_step)
        tot_b += b
        tot_s += sec
    val = tot_b / tot_s / 1e9
    return {"metric": METRIC, "value": round(val, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "dequant", "seq_len": int(wl.seq_lens[0]), "Hk": wl.Hk, "D": wl.D},
            "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": "each step: " + desc},
            "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["tiny", "batch", "outlier_long", "skewed", "outlier_ncu", "skewed_ncu",
                             "store", "dequant", "mq"])
    ap.add_argument("--impl", default="uq", choices=["uq", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the headline workload (no 'workloads' section)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "uq":
        args.warmup = 3
    rank, local, world = _dist_init()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_gpu(args, rank, local, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
