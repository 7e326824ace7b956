#!/usr/bin/env python3
"""Benchmark of the GDN layer core on GB300: prefill tokens/s and decode GB/s.

One step = one pass of the whole path on synthetic inputs of the pages'
Qwen3.5-4B geometry (Hq/Hk/Hv/D = 16/16/32/128):
  * gdn_prefill over one T=2048 sequence with the gated-RMSNorm epilogue
    (prep kernel + scan kernel), inputs rotated over 8 buffer sets so every
    step reads them from HBM (8 sets x ~67 MB of inputs >> 126 MB of L2);
  * gdn_decode of one token for 256 sequences, the 512 MiB fp32 state updated
    in place (larger than L2 by itself).
`value` is prefill tokens/s; the decode figures sit in the "decode" object.
CUDA events bracket each call inside the timed region, so each kernel family
gets its own measured time; the step time is the whole region / K.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torchrun: each rank processes its own replica (no data-path
collective), the timing is the max over ranks and `value` sums all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_deltanet_linear_08_gb300.inputs import (CASE_8x128, CASE_DECODE, CASE_T64, CASE_T2048,  # noqa: E402
                                                   CASE_VARLEN48, DecodeCase, DecodeSlotsCase, PrefillCase,
                                                   conv_channels, make_conv_inputs, make_decode_inputs,
                                                   make_decode_slots_inputs, make_prefill_inputs)

METRIC = "GDN prefill tokens/s & decode GB/s at Hv=32,D=128; % of tensor/HBM roofline"
PREFILL_FLOP_PER_TOKEN_HEAD = 10 * 64 * 128 + 6 * 128 * 128   # 180,224 (C=64 chunked count)
N_ROTATE = 8
KERNEL_SOURCES = ["gdn_api.cu", "gdn_conv.cu", "gdn_decode.cu", "gdn_prefill_prep.cu", "gdn_prefill_scan.cu",
                  "gdn_prefill_out.cu", "chunks.cuh", "common.cuh", "conv.cuh", "tc05.cuh", "kernels.h"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gated_deltanet_linear_08_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kind: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get(kind)


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def build_prefill_sets(dev, case: PrefillCase, n_sets: int):
    import gated_deltanet_linear_08_gb300 as gdn
    x = make_prefill_inputs(case)
    T, hk, hv, N = x["q"].shape[0], case.hk, case.hv, len(x["seqlens"])
    shared = {k: x[k].to(dev) for k in ("A_log", "dt_bias", "cu_seqlens", "norm_w")}
    sets = []
    for _ in range(n_sets):
        s = {k: x[k].to(dev) for k in ("q", "k", "v", "a", "b", "z")}
        s["out"] = torch.empty(T, hv, 128, dtype=torch.bfloat16, device=dev)
        s["fin"] = torch.empty(N, hv, 128, 128, dtype=torch.float32, device=dev)
        s["ws"] = gdn.alloc_workspace(N, T, hk, hv, dev)
        sets.append(s)
    return x, shared, sets


def packed_prefill_region(gdn, pre, stream, calls: int = 30, warmup: int = 3):
    """The T = 2048 prefill with q, k, v, z, b, a read in place from one packed
    projection buffer [T, 12352] (row order q | k | v | z | b | a): device
    time per call, rotating over the same number of buffer sets."""
    x, shared, sets = pre
    packed = []
    for st in sets:
        parts = [st["q"].flatten(1), st["k"].flatten(1), st["v"].flatten(1), st["z"].flatten(1), st["b"], st["a"]]
        buf = torch.cat(parts, dim=1).contiguous()
        offs, views = 0, {}
        for name, part in zip(("q", "k", "v", "z", "b", "a"), parts):
            views[name] = buf[:, offs:offs + part.shape[1]]
            offs += part.shape[1]
        for name in ("q", "k", "v", "z"):
            views[name] = views[name].unflatten(1, st[name].shape[1:])
        packed.append(dict(st, **views, buf=buf))
    for i in range(warmup):
        run_prefill(gdn, shared, packed[i % len(packed)], x["eps"], stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(calls):
        run_prefill(gdn, shared, packed[i % len(packed)], x["eps"], stream)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / calls


def run_prefill(gdn, shared, s, eps, stream):
    gdn.prefill(s["q"], s["k"], s["v"], s["a"], s["b"], shared["A_log"], shared["dt_bias"],
                shared["cu_seqlens"], init_state=None, z=s["z"], norm_w=shared["norm_w"],
                eps=eps, out=s["out"], final_state=s["fin"], workspace=s["ws"], stream=stream)


def build_decode(dev, case: DecodeCase):
    y = make_decode_inputs(DecodeCase(case.name, batch=case.batch, hk=case.hk, hv=case.hv,
                                      steps=1))
    d = {k: v.to(dev) for k, v in y["steps"][0].items()}
    d["A_log"], d["dt_bias"] = y["A_log"].to(dev), y["dt_bias"].to(dev)
    d["state"] = y["state"].to(dev)
    d["out"] = torch.empty(case.batch, case.hv, 128, dtype=torch.bfloat16, device=dev)
    return y, d


def run_decode(gdn, d, stream):
    gdn.decode(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["state"],
               out=d["out"], stream=stream)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (every rank gets it)."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every replica processes `units_per_rank` in the
    slowest rank's `ms`."""
    return world * units_per_rank / (ms * 1e-3)


def spread(ms):
    """p10, median and p90 of per-call times (nearest rank)."""
    s = sorted(ms)
    if not s:
        return None
    pick = lambda f: s[min(len(s) - 1, max(0, round(f * (len(s) - 1))))]
    return {"p10": pick(0.1), "median": statistics.median(s), "p90": pick(0.9)}


def timed_region(gdn, pre, dec, steps, warmup, stream, world):
    x, shared, sets = pre
    eps = x["eps"]
    for i in range(warmup):
        run_prefill(gdn, shared, sets[i % len(sets)], eps, stream)
        run_decode(gdn, dec, stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        e = ev[i]
        e[0].record(stream)
        run_prefill(gdn, shared, sets[i % len(sets)], eps, stream)
        e[1].record(stream)
        e[2].record(stream)
        run_decode(gdn, dec, stream)
        e[3].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev]
    return total_ms, pre_ms, dec_ms


def _layout(specs, align=256):
    """Byte offsets of tensors (shape, dtype) packed back to back, each start
    aligned to `align` bytes; returns (offsets, total bytes)."""
    offs, n = [], 0
    for shape, dt in specs:
        n = (n + align - 1) // align * align
        offs.append(n)
        n += int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
    return offs, (n + align - 1) // align * align


def _views(buf, specs, offs):
    """Typed views of `specs` into the uint8 buffer `buf` at `offs`."""
    out = []
    for (shape, dt), o in zip(specs, offs):
        nb = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
        out.append(buf[o:o + nb].view(dt).view(shape))
    return out


def e2e_region(gdn, x, dec_y, dev, steps, warmup, stream):
    """Same step through the public API with pinned host buffers, pipelined as
    a serving loop: every step copies all of its inputs host->device, runs
    both calls, and copies its results device->host, all inside the timed
    region.  A step's inputs sit packed in one pinned buffer and move in one
    copy, and so do its results (one copy each way per step); steps alternate
    between two device buffer sets, and the copies run on their own streams
    (one per direction), so step i+1's inputs and step i-1's results move
    while step i's kernels run; events order each buffer's reuse."""
    keys = ("q", "k", "v", "a", "b", "z")
    dkeys = ("q", "k", "v", "a", "b")
    st = dec_y["steps"][0]
    srcs = [x[k] for k in keys] + [st[k] for k in dkeys]
    in_specs = [(tuple(t.shape), t.dtype) for t in srcs]
    in_offs, in_bytes = _layout(in_specs)
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    for t, v in zip(srcs, _views(h_in, in_specs, in_offs)):
        v.copy_(t)
    shared = {k: x[k].to(dev) for k in ("A_log", "dt_bias", "cu_seqlens", "norm_w")}
    T, hv, N = x["q"].shape[0], x["hv"], len(x["seqlens"])
    ws = gdn.alloc_workspace(N, T, x["hk"], hv, dev)
    d_A, d_dt = dec_y["A_log"].to(dev), dec_y["dt_bias"].to(dev)
    d_state = dec_y["state"].to(dev)
    out_specs = [((T, hv, 128), torch.bfloat16), ((N, hv, 128, 128), torch.float32),
                 (tuple(st["v"].shape), torch.bfloat16)]
    out_offs, out_bytes = _layout(out_specs)
    bufs = []
    for _ in range(2):
        b = {"d_in": torch.empty(in_bytes, dtype=torch.uint8, device=dev),
             "d_out": torch.empty(out_bytes, dtype=torch.uint8, device=dev),
             "h_out": torch.empty(out_bytes, dtype=torch.uint8).pin_memory()}
        views = _views(b["d_in"], in_specs, in_offs)
        b["in"] = dict(zip(keys, views[:len(keys)]))
        b["din"] = dict(zip(dkeys, views[len(keys):]))
        b["out"], b["fin"], b["dout"] = _views(b["d_out"], out_specs, out_offs)
        b["loaded"], b["computed"], b["drained"] = (torch.cuda.Event() for _ in range(3))
        bufs.append(b)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    started = [False, False]

    def step(i):
        b = bufs[i % 2]
        with torch.cuda.stream(s_in):           # inputs of step i
            if started[i % 2]:
                s_in.wait_event(b["computed"])  # step i-2's kernels are done with them
            b["d_in"].copy_(h_in, non_blocking=True)
            b["loaded"].record(s_in)
        with torch.cuda.stream(stream):         # kernels of step i
            stream.wait_event(b["loaded"])
            if started[i % 2]:
                stream.wait_event(b["drained"])  # step i-2's results are out
            d = b["in"]
            gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], shared["A_log"], shared["dt_bias"],
                        shared["cu_seqlens"], z=d["z"], norm_w=shared["norm_w"], eps=x["eps"],
                        out=b["out"], final_state=b["fin"], workspace=ws, stream=stream)
            dd = b["din"]
            gdn.decode(dd["q"], dd["k"], dd["v"], dd["a"], dd["b"], d_A, d_dt, d_state, out=b["dout"],
                       stream=stream)
            b["computed"].record(stream)
        with torch.cuda.stream(s_out):          # results of step i
            s_out.wait_event(b["computed"])
            b["h_out"].copy_(b["d_out"], non_blocking=True)
            b["drained"].record(s_out)
        started[i % 2] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(warmup, warmup + steps):
        step(i)
    s_in.wait_stream(s_out)
    e.record(s_in)
    torch.cuda.synchronize()
    # the last step's prefill results, as they reached the host, equal a plain
    # call on the same inputs (the packed views hold what they should)
    last = bufs[(warmup + steps - 1) % 2]
    h_out, h_fin, _ = _views(last["h_out"], out_specs, out_offs)
    ref_out = torch.empty_like(last["out"])
    ref_fin = torch.empty_like(last["fin"])
    gdn.prefill(*(x[k].to(dev) for k in ("q", "k", "v", "a", "b")), shared["A_log"], shared["dt_bias"],
                shared["cu_seqlens"], z=x["z"].to(dev), norm_w=shared["norm_w"], eps=x["eps"],
                out=ref_out, final_state=ref_fin, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    assert torch.equal(h_out, ref_out.cpu()) and torch.equal(h_fin, ref_fin.cpu()), "end-to-end results differ"
    return a.elapsed_time(e) / steps, in_bytes, out_bytes


# ---------------------------------------------------------------------------
# CPU legs: the fp64 oracle as it stands, on the host cores
# ---------------------------------------------------------------------------
def _oracle_prefill_sample(T: int, nthreads: int = 0):
    """Oracle prefill on the first T tokens of the T=2048 workload (all 32
    heads), on `nthreads` host threads (0: all cores)."""
    import oracle
    from gated_deltanet_linear_08_gb300.inputs import to_f64
    x = make_prefill_inputs(CASE_T2048)
    cu = torch.tensor([0, T], dtype=torch.int32).numpy()
    f = {k: to_f64(x[k]) for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "z", "norm_w")}
    for k in ("q", "k", "v", "a", "b", "z"):
        f[k] = f[k][:T]

    def run():
        oracle.prefill(cu, f["q"], f["k"], f["v"], f["a"], f["b"], f["A_log"], f["dt_bias"],
                       None, f["z"], f["norm_w"], eps=x["eps"], nthreads=nthreads or os.cpu_count())
    return run


def _oracle_decode_sample(B: int):
    import numpy as np

    import oracle
    from gated_deltanet_linear_08_gb300.inputs import to_f64
    y = make_decode_inputs(DecodeCase("cpu", batch=B, steps=1))
    st = {k: to_f64(v) for k, v in y["steps"][0].items()}
    S = np.ascontiguousarray(to_f64(y["state"]))
    A_log, dt = to_f64(y["A_log"]), to_f64(y["dt_bias"])

    def run():
        oracle.decode_step(st["q"], st["k"], st["v"], st["a"], st["b"], A_log, dt, S,
                           nthreads=os.cpu_count())
    return run


def decode_state_bytes(batch: int, hv: int = 32, hk: int = 16, tokens: int = 1) -> int:
    """Algorithmic bytes of one decode call: every fp32 state read and written
    once, plus each token's inputs and bf16 output."""
    state = batch * hv * 128 * 128 * 4 * 2
    io = tokens * batch * (2 * hk * 128 * 2 + hv * 128 * 2 + 2 * hv * 2 + hv * 128 * 2)
    return state + io


SLOTS_CASE = DecodeSlotsCase("decode_slots_B256_T4", batch=256, tokens=4, slots=256)


def decode_slots_region(gdn, dev, stream, calls: int = 50, warmup: int = 5):
    """Multi-token decode over a slot pool (256 sequences x 4 draft tokens, a
    random slot permutation of a 256-slot pool): device time per call."""
    y = make_decode_slots_inputs(SLOTS_CASE)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in y.items()}
    out = torch.empty(SLOTS_CASE.batch, SLOTS_CASE.tokens, SLOTS_CASE.hv, 128, dtype=torch.bfloat16, device=dev)

    def call():
        gdn.decode_slots(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["pool"],
                         state_idx=d["state_idx"], out=out, stream=stream)
    for _ in range(warmup):
        call()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(calls):
        call()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / calls


def time_calls(call, calls: int, warmup: int, stream) -> float:
    """Device time per call of call(i) on `stream`, by CUDA events."""
    for i in range(warmup):
        call(i)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(calls):
        call(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / calls


def prefill_bytes(T: int, N: int, hk: int, hv: int, gated: bool, init: bool) -> int:
    """Algorithmic HBM bytes of one prefill call: q, k, v, a, b read and the
    bf16 output written once per token (z too with the epilogue), the final
    states written and the initial states read once per sequence."""
    per_tok = 2 * hk * 256 + hv * 256 + 2 * hv * 2 + hv * 256 + (hv * 256 if gated else 0)
    return T * per_tok + N * hv * 128 * 128 * 4 * (2 if init else 1)


L2_FLUSH_BYTES = 256 << 20   # twice the 129 MB L2


def prefill_config_region(gdn, case: PrefillCase, dev, stream, peaks, calls: int = 20, warmup: int = 3):
    """One of the other prefill workloads: the device time of each call by
    CUDA events on the launching stream, with L2 flushed between calls
    (outside the events), so every call reads its inputs from HBM."""
    x = make_prefill_inputs(case)
    d = {k: (None if x[k] is None else x[k].to(dev)) for k in
         ("q", "k", "v", "a", "b", "A_log", "dt_bias", "init_state", "cu_seqlens", "z", "norm_w")}
    T, N, hk, hv = x["q"].shape[0], len(x["seqlens"]), case.hk, case.hv
    out = torch.empty(T, hv, 128, dtype=torch.bfloat16, device=dev)
    fin = torch.empty(N, hv, 128, 128, dtype=torch.float32, device=dev)
    ws = gdn.alloc_workspace(N, T, hk, hv, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def call():
        gdn.prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["cu_seqlens"],
                    init_state=d["init_state"], z=d["z"], norm_w=d["norm_w"], eps=x["eps"], out=out,
                    final_state=fin, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    mean = sum(ms) / len(ms)
    flops = T * hv * PREFILL_FLOP_PER_TOKEN_HEAD
    nbytes = prefill_bytes(T, N, hk, hv, case.gated_norm, case.init_state)
    return {"workload": f"{N} sequence(s), {T} tokens, Hk/Hv = {hk}/{hv}"
                        + (", initial states" if case.init_state else "")
                        + (", gated RMSNorm" if case.gated_norm else ""),
            "ms_per_call": mean, "ms_spread": spread(ms), "tokens_per_s": T / (mean * 1e-3),
            "tensor_frac": flops / (mean * 1e-3) / 1e12 / peaks["bf16"],
            "hbm_frac": nbytes / (mean * 1e-3) / 1e9 / peaks["hbm"],
            "algorithmic_flop": flops, "algorithmic_bytes": nbytes,
            "l2": "flushed between calls (256 MiB written outside the events)"}


CONV_WIDTH = 4


def conv_prefill_region(gdn, pre, stream, calls: int = 30, warmup: int = 3):
    """The T = 2048 prefill with the width-4 causal conv + SiLU ahead of
    the core (weights [8192, 4], a carried conv state in and out)."""
    x, shared, sets = pre
    C = conv_channels(16, x["hv"])
    cv = make_conv_inputs(C, CONV_WIDTH, 1, seed=1)
    w = cv["weight"].to(sets[0]["q"].device)
    states = [cv["state"].to(w.device) for _ in sets]
    outs = [torch.empty_like(st) for st in states]
    wss = [gdn.alloc_workspace(1, x["q"].shape[0], 16, x["hv"], w.device, conv=True) for _ in sets]

    def call(i):
        s = sets[i % len(sets)]
        gdn.prefill(s["q"], s["k"], s["v"], s["a"], s["b"], shared["A_log"], shared["dt_bias"],
                    shared["cu_seqlens"], init_state=None, z=s["z"], norm_w=shared["norm_w"], eps=x["eps"],
                    out=s["out"], final_state=s["fin"], workspace=wss[i % len(sets)], stream=stream, conv_weight=w,
                    conv_state=states[i % len(sets)], conv_state_out=outs[i % len(sets)])
    return time_calls(call, calls, warmup, stream)


def conv_decode_region(gdn, dec, stream, in_place: bool, calls: int = 50, warmup: int = 5):
    """Batch-256 decode with the width-4 conv and conv-state pools [256, 3,
    8192]: two pools used in turn (the decode kernel writes the new states),
    or one pool rolled in place by the follow-up kernel."""
    B, hv = dec["q"].shape[0], dec["v"].shape[1]
    cv = make_conv_inputs(conv_channels(16, hv), CONV_WIDTH, B, seed=2)
    w = cv["weight"].to(dec["q"].device)
    pools = [cv["state"].to(w.device), cv["state"].to(w.device)]
    tok = {n: dec[n].unsqueeze(1) for n in ("q", "k", "v", "a", "b")}
    out = dec["out"].unsqueeze(1)

    def call(i):
        src = pools[i % 2]
        dst = src if in_place else pools[(i + 1) % 2]
        gdn.decode_slots(tok["q"], tok["k"], tok["v"], tok["a"], tok["b"], dec["A_log"], dec["dt_bias"],
                         dec["state"], out=out, stream=stream, conv_weight=w, conv_state=src, conv_state_out=dst)
    return time_calls(call, calls, warmup, stream)


def _repeat_for(fn, seconds: float, max_reps: int = 1000):
    """Run fn until `seconds` of wall time have passed; (reps, seconds per rep)."""
    fn()   # warm (page-in, thread pool)
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= max_reps:
            return reps, el / reps


def cpu_baseline(seconds: float = 10.0):
    """The fp64 oracle as it stands on the host cores: the whole T=2048
    prefill repeated for about `seconds`, and the batch-256 decode step
    repeated for a third of that."""
    reps, tp = _repeat_for(_oracle_prefill_sample(2048), seconds)
    dreps, td = _repeat_for(_oracle_decode_sample(CASE_DECODE.batch), seconds / 3)
    # one core: the first 512 tokens (the recurrence costs the same per token)
    sreps, ts = _repeat_for(_oracle_prefill_sample(512, nthreads=1), seconds / 3)
    return {"value": 2048 / tp, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"fp64 oracle, the full T=2048 prefill (32 heads, gated norm) x {reps} "
                      f"({reps * tp:.1f} s); decode: the 256-sequence step x {dreps} ({dreps * td:.1f} s)",
            "seconds": round(reps * tp, 2),
            "decode": {"value": decode_state_bytes(CASE_DECODE.batch) / td / 1e9, "unit": "GB/s",
                       "tokens_per_s": CASE_DECODE.batch / td, "seconds": round(dreps * td, 2)},
            "single_core": {"value": 512 / ts, "unit": "tokens/s", "cores": 1,
                            "sample": f"the first 512 tokens (32 heads, gated norm) x {sreps}",
                            "seconds": round(sreps * ts, 2)}}


def reference_arm(args, rank):
    if rank != 0:
        return
    T_SAMPLE, B_SAMPLE = 64, 8
    pre, dec = _oracle_prefill_sample(T_SAMPLE), _oracle_decode_sample(B_SAMPLE)
    for _ in range(args.warmup):
        pre(); dec()
    tp = td = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = time.perf_counter(); pre(); b = time.perf_counter(); dec(); c = time.perf_counter()
        tp += b - a
        td += c - b
    total = time.perf_counter() - t0
    value = T_SAMPLE * args.steps / tp
    dec_gbs = decode_state_bytes(B_SAMPLE) * args.steps / td / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_per_step":
                   f"oracle prefill of the first {T_SAMPLE} tokens (32 heads, gated norm) "
                   f"+ oracle decode of {B_SAMPLE} sequences"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": f"{T_SAMPLE}-token prefill + "
                         f"{B_SAMPLE}-sequence decode per step"},
        "decode": {"value": dec_gbs, "unit": "GB/s"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


WORKLOAD = ("GDN core, Hq/Hk/Hv/D = 16/16/32/128: prefill of one T=2048 sequence with "
            "gated-RMSNorm epilogue, zero initial state; decode of 256 sequences x 1 token, "
            "fp32 states updated in place")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return

    import gated_deltanet_linear_08_gb300 as gdn
    from gated_deltanet_linear_08_gb300 import build as gbuild
    gbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    gdn.load()

    peaks = load_peaks()
    pre = build_prefill_sets(dev, CASE_T2048, N_ROTATE)
    dec_y, dec = build_decode(dev, CASE_DECODE)
    stream = torch.cuda.Stream(device=dev)
    x = pre[0]
    T, hv = x["q"].shape[0], x["hv"]

    with ClockSampler(local) as clk:
        total_ms, pre_ms, dec_ms = timed_region(gdn, pre, dec, args.steps, args.warmup, stream,
                                                world)
    assert gdn.check_device_status() == 0
    total_ms = max_over_ranks(total_ms, world)
    pre_mean = max_over_ranks(sum(pre_ms) / len(pre_ms), world)
    dec_mean = max_over_ranks(sum(dec_ms) / len(dec_ms), world)

    flops = T * hv * PREFILL_FLOP_PER_TOKEN_HEAD
    tflops = flops / (pre_mean * 1e-3) / 1e12
    pre_bytes = T * (2 * 16 * 256 + 2 * hv * 256 + 2 * hv * 2 + hv * 256) + hv * 128 * 128 * 4
    dbytes = decode_state_bytes(CASE_DECODE.batch)
    dec_gbs = dbytes / (dec_mean * 1e-3) / 1e9

    line = {
        "metric": METRIC,
        "value": job_rate(T, world, pre_mean),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world,
                   "seq_len": T, "decode_batch": CASE_DECODE.batch * world,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"prefill inputs rotated over {N_ROTATE} buffer sets (> L2); "
                         "decode state 512 MiB (> L2)"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16"],
                     "unit": "TFLOP/s", "frac": tflops / peaks["bf16"],
                     "traffic": ncu_traffic("prefill"),
                     "kernel": "gdn_prefill call (prep, scan and output kernels)",
                     "peak_kind": f"{peaks['src']} bf16 burst",
                     "work": f"{flops} algorithmic flop per call "
                             f"({PREFILL_FLOP_PER_TOKEN_HEAD} per token per value head)"},
        "prefill": {"ms_per_call": pre_mean, "ms_spread": spread(pre_ms), "algorithmic_bytes": pre_bytes,
                    "hbm_gbs": pre_bytes / (pre_mean * 1e-3) / 1e9,
                    "hbm_frac": pre_bytes / (pre_mean * 1e-3) / 1e9 / peaks["hbm"],
                    "workspace_bytes": gdn.workspace_bytes(1, T, 16, hv)},
        "decode": {"value": world * dec_gbs, "unit": "GB/s", "ms_per_call": dec_mean, "ms_spread": spread(dec_ms),
                   "tokens_per_s": world * CASE_DECODE.batch / (dec_mean * 1e-3),
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm"],
                                "unit": "GB/s", "frac": dec_gbs / peaks["hbm"],
                                "frac_of_nominal_8tbs": dec_gbs / 8000.0,
                                "traffic": ncu_traffic("decode"),
                                "kernel": "decode_kernel",
                                "peak_kind": f"{peaks['src']} HBM copy",
                                "work": f"{dbytes} algorithmic bytes per call"}},
        "gpu_launches": 4 * args.steps,
        "clocks": clk.summary(),
    }
    line["prefill_configs"] = {}
    for case in (CASE_T64, CASE_8x128, CASE_VARLEN48):
        r = prefill_config_region(gdn, case, dev, stream, peaks)
        r["ms_per_call"] = max_over_ranks(r["ms_per_call"], world)
        line["prefill_configs"][case.name] = r
    pk_ms = max_over_ranks(packed_prefill_region(gdn, pre, stream), world)
    line["prefill_packed_inputs"] = {
        "workload": "the same T=2048 prefill, inputs read in place from a packed [T, 12352] projection buffer",
        "ms_per_call": pk_ms, "tokens_per_s": world * T / (pk_ms * 1e-3)}
    sl_ms = max_over_ranks(decode_slots_region(gdn, dev, stream), world)
    sl_bytes = decode_state_bytes(SLOTS_CASE.batch, tokens=SLOTS_CASE.tokens)
    line["decode_slots"] = {
        "workload": "256 sequences x 4 draft tokens against a 256-slot state pool (random slot permutation)",
        "value": world * sl_bytes / (sl_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_call": sl_ms,
        "tokens_per_s": world * SLOTS_CASE.batch * SLOTS_CASE.tokens / (sl_ms * 1e-3),
        "hbm_frac": sl_bytes / (sl_ms * 1e-3) / 1e9 / peaks["hbm"]}
    cp_ms = max_over_ranks(conv_prefill_region(gdn, pre, stream), world)
    cd_ms = max_over_ranks(conv_decode_region(gdn, dec, stream, in_place=False), world)
    cdi_ms = max_over_ranks(conv_decode_region(gdn, dec, stream, in_place=True), world)
    conv_state_b = CASE_DECODE.batch * (CONV_WIDTH - 1) * conv_channels(16, hv) * 2
    cd_bytes = dbytes + 2 * conv_state_b
    line["conv"] = {
        "workload": "causal conv1d (width 4) + SiLU on q | k | v ahead of the core (conv pass, then the core)",
        "prefill_ms_per_call": cp_ms, "prefill_tokens_per_s": world * T / (cp_ms * 1e-3),
        "prefill_overhead_vs_plain": cp_ms / pre_mean - 1.0,
        "decode_ms_per_call": cd_ms, "decode_gbs": cd_bytes / (cd_ms * 1e-3) / 1e9,
        "decode_hbm_frac": cd_bytes / (cd_ms * 1e-3) / 1e9 / peaks["hbm"],
        "decode_overhead_vs_plain": cd_ms / dec_mean - 1.0,
        "decode_pools": "two conv-state pools used in turn (state_out apart from state_in)",
        "decode_in_place_ms_per_call": cdi_ms,
        "decode_in_place_overhead_vs_plain": cdi_ms / dec_mean - 1.0}
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_region(gdn, x, dec_y, dev, max(10, min(args.steps, 200)),
                                      3, stream)
        e2e_ms = max_over_ranks(e2e_ms, world)
        line["e2e"] = {"value": job_rate(T, world, e2e_ms), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms,
                       "pipeline": "each step's inputs packed in one pinned buffer and copied in one "
                                   "host->device copy, its results in one device->host copy; two device "
                                   "buffer sets; the copies run on their own streams and overlap the "
                                   "neighbouring steps' kernels"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
