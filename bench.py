#!/usr/bin/env python3
"""Throughput of the DFlash2 draft-head hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
the grouped dynamic depthwise causal convolution, the projection of every
position's hidden state, and the edge scores with the per-predecessor argmax.
The default workload is the batched verification regime (256 sequences x 16
positions, d = C = 5120, T = 4, G = 40, R = 128, V = 151936, K = 16).

Prints ONE JSON line (rank 0).  The metric is draft positions per second
(conv positions of all ranks / max-over-ranks time); the dominant kernel's
achieved HBM bandwidth is reported against the measured peak.

  python bench.py [--gpus N --steps K --warmup W --workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DFlash2 conv+selector draft positions/sec; achieved HBM GB/s vs GB300 peak"
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FLUSH_BYTES = 256 << 20
P_MIN = 0.05  # draft-probability cut of the chain readout line

# DRAM bytes per launch of the dominant kernel from an ncu capture, keyed by the
# sha256 of the kernel source they were taken on (null when the source changed).
TRAFFIC = {
    ("batched_256x16_d5120", "dynconv"): {
        "sha": "c48948d39e2a8c96f8f4fcd2efbeb99d00967436575f467308906f108b4fb11e",
        "bytes": 51194880 + 3361280,  # dram__bytes_read.sum + dram__bytes_write.sum
    },
    # captured on 512 rows (same kernel, same V and K), scaled by 4096 / 512: every row
    # streams once, so DRAM traffic grows in proportion to the rows
    ("batched_256x16_d5120", "topk"): {
        "sha": "44bcef28a9e26a4fb49140d8ca8d19c39eef514ce542cdf321497360a4e547d3",
        "bytes": 8 * (311339776 + 3530496),
    },
    ("batched_256x16_d5120", "select"): {
        "sha": "6612f58bcc72d04450b131bd2958dbfd202b8042e9e5b9ea71329c420c3e2c45",
        "bytes": 69798656 + 977408,
    },
    ("batched_256x16_d5120", "dynconv_predicted"): {
        "sha": "8b1254453ff647de614a550e6b7a3a920bd343bed6d783b0234df397d6484d6e",
        "bytes": 52569856 + 3127296,
    },
}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="dflash2", choices=["dflash2", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="oracle time the reference arm spreads over warm-up and timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the steps of the other four workloads")
    return ap.parse_args()


def _env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(w0, rank):
    """The workload a rank runs: same shapes, its own sequences (seed offset by rank)."""
    return dataclasses.replace(w0, seed=w0.seed + 1000 * rank)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (a measurement reduction, not a data path)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def _workload(name):
    from dflash2_draft_head_gb300.workloads import BENCH_WORKLOAD, BY_NAME
    return BY_NAME[name] if name else BENCH_WORKLOAD


def _config(w, world):
    return {"workload": w.name, "S": w.S, "n": w.n, "C": w.C, "T": w.T, "G": w.G, "d": w.d,
            "R": w.R, "V": w.V, "K": w.K, "selector_S": w.S_sel, "selector_n": w.n_sel,
            "in_dtype": w.dtype, "out_dtype": w.dtype,
            "l2": f"flushed between timed steps ({FLUSH_BYTES >> 20} MiB write, then "
                  f"{FLUSH_BYTES >> 20} MiB read)",
            "parallelism": f"replicas x{world} (independent sequences per GPU)"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def _bytes(w):
    """Algorithmic bytes (each element streamed or gathered once, plus outputs)."""
    b = 2 if w.dtype == "bf16" else 4
    conv = (w.S * w.n * w.C * (b + b) + w.S * w.n * w.T * w.G * b + w.S * (w.T - 1) * w.C * b
            + w.T * w.C * b)
    P = w.S_sel * w.n_sel
    proj = P * w.d * b + w.R * w.d * b + P * w.R * 4
    proj_flops = 2.0 * P * w.d * w.R
    E = w.S_sel * max(w.n_sel - 1, 0)
    edges = E * (2 * w.K * w.R * b + 4 * w.R + 20 * w.K)
    return conv, proj, proj_flops, edges


# ---------------------------------------------------------------- oracle (CPU)

class OraclePool:
    """Float64 copies of the workload's inputs, cut into units of up to 16 sequences."""

    def __init__(self, w, max_units=16):
        import numpy as np
        from dflash2_draft_head_gb300 import synth
        self.w = w
        ub = min(w.S, 16)
        self.ub = ub
        self.units = []
        n_conv = min(w.n, 4096)
        self.n_conv = n_conv
        base = synth.normal_whole(w.seed, "base", (w.T, w.C), math.sqrt(1.0 / w.T), w.dtype)
        cb = synth.codebooks(w)
        self.base = base.numpy().astype(np.float64)
        self.W = cb["W"].numpy().astype(np.float64)
        self.A = cb["A"].numpy().astype(np.float64)
        self.B = cb["B"].numpy().astype(np.float64)
        sel = synth.selector_inputs(w)
        h = sel["h"].reshape(w.S_sel, w.n_sel, w.d)
        for u0 in range(0, min(w.S, ub * max_units), ub):
            ss = range(u0, min(w.S, u0 + ub))
            x = np.stack([synth.normal_rows(w.seed, "x", s, 0, n_conv, (w.C,), 1.0, w.dtype,
                                            w.n).numpy() for s in ss]).astype(np.float64)
            hist = np.stack([synth.normal_rows(w.seed, "hist", s, 0, w.T - 1, (w.C,), 1.0,
                                               w.dtype, w.T - 1).numpy() for s in ss]
                            ).astype(np.float64)
            delta = np.stack([synth.normal_rows(w.seed, "delta", s, 0, n_conv, (w.T, w.G),
                                                math.sqrt(0.1 / w.T), w.dtype, w.n).numpy()
                              for s in ss]).astype(np.float64)
            s0, s1 = min(u0, w.S_sel), min(u0 + ub, w.S_sel)
            self.units.append(dict(
                x=x, hist=hist, delta=delta,
                h=h[s0:s1].reshape(-1, w.d).numpy().astype(np.float64),
                ids=sel["cand_ids"][s0:s1].numpy(),
                unary=sel["unary"][s0:s1].numpy().astype(np.float64),
                positions=len(ss) * n_conv))

    def run(self, j):
        import oracle
        u = self.units[j % len(self.units)]
        oracle.dynconv(u["x"], u["hist"], self.base, u["delta"])
        if u["ids"].shape[0] > 0:
            oracle.select(u["h"], self.W, u["ids"], self.A, self.B, u["unary"],
                          want_edges=False)
        return u["positions"]

    def describe(self, reps):
        w = self.w
        return (f"{reps} oracle passes (dynconv + project + edges/argmax) over units of "
                f"{self.ub} sequences x {self.n_conv} positions of {w.name} "
                f"(selector on {w.n_sel} positions per sequence), fp64")


def cpu_baseline(w, seconds):
    import oracle
    oracle.build()
    pool = OraclePool(w)
    pool.run(0)  # warm the code and pages
    t0 = time.perf_counter()
    pos = 0
    reps = 0
    while True:
        pos += pool.run(reps)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 100000:
            break
    return {"value": pos / el, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": pool.describe(reps), "seconds": round(el, 3)}


def run_reference(args):
    rank, world, _ = _env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = _workload(args.workload)
    pool = OraclePool(w)
    pool.run(0)
    t0 = time.perf_counter()
    pool.run(0)
    t_unit = max(time.perf_counter() - t0, 1e-4)
    total_budget = max(float(args.ref_seconds), 0.0)
    units_per_step = max(1, int(total_budget / max(args.steps + args.warmup, 1) / t_unit))
    for k in range(args.warmup):
        for j in range(units_per_step):
            pool.run(k * units_per_step + j)
    pos = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        for j in range(units_per_step):
            pos += pool.run(k * units_per_step + j)
    el = time.perf_counter() - t0
    v = pos / el
    cores = oracle.max_threads()
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * el / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: {units_per_step} units; "
                                       + pool.describe(units_per_step * args.steps)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- host link

def _host_link(pin, dst, copy_streams, split, stream, reps=5):
    """Pinned host -> device copy rate of one step's inputs (the e2e loop's
    tensors and copy streams), with no kernel running: all tensors on one
    stream, then split over the two copy streams as the e2e loop splits them."""
    import torch

    nbytes = sum(v.numel() * v.element_size() for v in pin.values())

    def run(groups):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for cst in copy_streams[:len(groups)]:
            cst.wait_event(e0)
        for _ in range(reps):
            for cst, names in zip(copy_streams, groups):
                with torch.cuda.stream(cst):
                    for k in names:
                        dst[k].copy_(pin[k], non_blocking=True)
        for cst in copy_streams[:len(groups)]:
            ev = torch.cuda.Event()
            ev.record(cst)
            stream.wait_event(ev)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    one = [sorted(pin)]
    run(one)
    t1 = run(one)
    t2 = run(split)
    return {"bytes": nbytes, "reps": reps, "GB/s_1stream": nbytes * reps / t1 / 1e6,
            "GB/s_2streams": nbytes * reps / t2 / 1e6}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        self.gpu_id = gpu_id

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        time.sleep(0.2)
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

class L2Flush:
    """Evicts L2 between timed steps: write one buffer larger than L2, then read
    another, so that L2 ends full of clean lines (no write-back is left for the
    next timed kernel to pay)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def zero_(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)

class _NoFlush:
    """Stands in for the L2 flush where a warm-cache variant is timed."""

    def zero_(self):
        pass


def _input_digests(tensors):
    """SHA-256 of every host input tensor's bytes (storage dtype), for reproducibility."""
    import torch
    out = {}
    for k, v in tensors.items():
        t = v.contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)  # numpy has no bf16: hash the raw 16-bit words
        out[k] = hashlib.sha256(t.numpy().tobytes()).hexdigest()
    return out


def _event_record_external():
    """cudaEventRecordWithFlags(..., cudaEventRecordExternal) of the CUDA runtime torch
    loaded (timing events inside a captured graph), or None."""
    import ctypes
    path = None
    try:
        for line in open("/proc/self/maps"):
            if "libcudart.so" in line:
                path = line.split()[-1]
                break
    except OSError:
        return None
    if path is None:
        return None
    try:
        f = ctypes.CDLL(path).cudaEventRecordWithFlags
    except (OSError, AttributeError):
        return None
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    f.restype = ctypes.c_int
    return f


def _call(f, a, L):
    if f(*a):
        raise RuntimeError(L.dflash2_last_error().decode())


def _timed_graph(K, stream, flush, calls, record_ext, L, per_graph=50, ends_only=False):
    """K steps replayed from CUDA graphs.  Each step: L2 flush, then the calls in
    order, with a timing event (recorded as a graph node) before the first call
    and after every call.  Returns, per call, the list of per-step times (ms).
    With ends_only the events bracket the whole step (one before the first call,
    one after the last) and a single list of step times is returned."""
    import ctypes

    import torch
    sp = ctypes.c_void_p(stream.cuda_stream)
    nc = len(calls)
    if ends_only:
        seq = calls

        def run_all():
            for f, a in seq:
                _call(f, a, L)
        calls = [(None, run_all)]
        nc = 1
    times = [[] for _ in range(nc)]
    done = 0
    graphs = {}
    while done < K:
        M = min(per_graph, K - done)
        if M not in graphs:
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(M)]
            for e4 in ev:
                for e in e4:
                    e.record(stream)  # materialise the event handles
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for m in range(M):
                    flush.zero_()
                    for j, (f, a) in enumerate(calls):
                        if record_ext(ctypes.c_void_p(ev[m][j].cuda_event), sp, 1):
                            raise RuntimeError("event record in capture failed")
                        if f is None:
                            a()
                        else:
                            _call(f, a, L)
                    if record_ext(ctypes.c_void_p(ev[m][nc].cuda_event), sp, 1):
                        raise RuntimeError("event record in capture failed")
            graphs[M] = (g, ev)
        g, ev = graphs[M]
        g.replay()
        stream.synchronize()
        for e in ev:
            for j in range(nc):
                times[j].append(e[j].elapsed_time(e[j + 1]))
        done += M
    return times[0] if ends_only else times


def _timed_eager(K, stream, flush, calls, L, ends_only=False):
    """K eagerly launched steps (fallback when graph timing events are unavailable)."""
    import torch
    nc = 1 if ends_only else len(calls)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(K)]
    torch.cuda._sleep(20_000_000)  # let the host queue ahead of the device
    for k in range(K):
        flush.zero_()
        for j, (f, a) in enumerate(calls):
            if not ends_only or j == 0:
                ev[k][0 if ends_only else j].record(stream)
            _call(f, a, L)
        ev[k][nc].record(stream)
    stream.synchronize()
    t = [[e[j].elapsed_time(e[j + 1]) for e in ev] for j in range(nc)]
    return t[0] if ends_only else t


def _back_to_back_us(stream, flush, calls, L, reps=20, iters=10):
    """Per-call device time of `calls` when launched back to back from a CUDA graph:
    a graph of `reps` (L2 flush + calls) minus a graph of `reps` flushes, each timed
    with two CUDA events around `iters` replays (median); no timing event sits
    between the calls, so the launch gaps the per-call events add are left out."""
    import torch

    def graph_us(cl):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                flush.zero_()
                for f, a in cl:
                    _call(f, a, L)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        g.replay()
        ts = []
        for _ in range(iters):
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            ts.append(e0.elapsed_time(e1))
        return 1000.0 * statistics.median(ts) / reps
    return graph_us(calls) - graph_us([])


def _timer(stream, record_ext, L):
    """timer(K, flush, calls, ends_only=False): the graph timer when timing events
    can be recorded inside a capture, else eager launches."""
    def timer(K, flush, calls, ends_only=False):
        if record_ext is not None:
            return _timed_graph(K, stream, flush, calls, record_ext, L, ends_only=ends_only)
        return _timed_eager(K, stream, flush, calls, L, ends_only=ends_only)
    return timer


def _select_fused(L, w):
    """Whether dflash2_select runs these shapes as one kernel (dflash2_select_plan)."""
    import ctypes
    out = (ctypes.c_int * 4)()
    code = 1 if w.dtype == "bf16" else 0
    if L.dflash2_select_plan(w.S_sel, w.n_sel, w.d, w.K, w.R, code, out):
        raise RuntimeError(L.dflash2_last_error().decode())
    return {"fused": bool(out[0]), "cluster_size": out[1], "clusters": out[2],
            "rows_per_block": out[3]}


def workload_leg(name, dev, stream, flush, timer, L, steps):
    """The step (dynconv + select) of another workload: the whole step between two
    events, and each call on its own, L2 flushed before every step."""
    import ctypes

    import torch

    from dflash2_draft_head_gb300 import synth
    w = _workload(name)
    bt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ci = synth.conv_inputs(w)
    cb = synth.codebooks(w)
    si = synth.selector_inputs(w)

    def d(t, dt=bt):
        return t.to(dt).to(dev).contiguous()
    x, hist, base, delta = d(ci["x"]), d(ci["hist"]), d(ci["base"]), d(ci["delta"])
    h, W, A, B = d(si["h"]), d(cb["W"]), d(cb["A"]), d(cb["B"])
    ids, un = si["cand_ids"].to(dev), si["unary"].to(dev)
    del ci, cb, si
    out = torch.empty((w.S, w.n, w.C), dtype=bt, device=dev)
    P = w.S_sel * w.n_sel
    E = w.S_sel * max(w.n_sel - 1, 0)
    u = torch.empty((P, w.R), dtype=torch.float32, device=dev)
    slot = torch.empty((max(E, 1), w.K), dtype=torch.int32, device=dev)
    score = torch.empty((max(E, 1), w.K), dtype=torch.float32, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    vp = ctypes.c_void_p
    sp = vp(stream.cuda_stream)
    code = 1 if w.dtype == "bf16" else 0

    def ptr(t):
        return vp(t.data_ptr())
    conv_args = (ptr(x), ptr(hist), ptr(base), ptr(delta), ptr(out), w.S, w.n, w.C, w.T, w.G,
                 code, code, sp)
    sel_args = (ptr(h), ptr(W), ptr(ids), ptr(A), ptr(B), ptr(un), w.S_sel, w.n_sel, w.d, w.K,
                w.R, w.V, code, ptr(u), None, ptr(slot), ptr(score), ptr(flag), sp)
    calls = [(L.dflash2_dynconv, conv_args), (L.dflash2_select, sel_args)]
    for _ in range(3):
        flush.zero_()
        for f, a in calls:
            _call(f, a, L)
    torch.cuda.synchronize()
    t_step = timer(steps, flush, calls, ends_only=True)
    t_conv, t_sel = timer(steps, flush, calls)
    # the two-kernel selector on the same shapes (what select runs when not fused)
    proj_args = (ptr(h), ptr(W), ptr(u), P, w.d, w.R, code, sp)
    edge_args = (ptr(ids), ptr(u), ptr(A), ptr(B), ptr(un), w.S_sel, w.n_sel, w.K, w.R, w.V, code,
                 None, ptr(slot), ptr(score), ptr(flag), sp)
    t_pair = timer(steps, flush, [(L.dflash2_project, proj_args), (L.dflash2_edges, edge_args)],
                   ends_only=True)
    torch.cuda.synchronize()
    if int(flag.item()) != 0:
        raise RuntimeError(f"device error flag set in the {name} leg")
    hbm = _peaks()[0]
    conv_b, proj_b, proj_f, edge_b = _bytes(w)
    step_us = 1000.0 * statistics.median(t_step)
    conv_us = 1000.0 * statistics.median(t_conv)
    sel_us = 1000.0 * statistics.median(t_sel)
    plan = _select_fused(L, w)
    return {
        "dtype": w.dtype, "steps": steps, "S": w.S, "n": w.n, "C": w.C, "T": w.T, "G": w.G,
        "R": w.R, "V": w.V, "K": w.K, "selector_S": w.S_sel, "selector_n": w.n_sel,
        "step_us": step_us, "positions_per_s": w.S * w.n / (step_us * 1e-6),
        "step_bytes": conv_b + proj_b + edge_b,
        "step_frac_hbm": (conv_b + proj_b + edge_b) / step_us / 1e3 / hbm,
        "dynconv": {"us": conv_us, "bytes": conv_b, "GB/s": conv_b / conv_us / 1e3,
                    "frac_hbm": conv_b / conv_us / 1e3 / hbm},
        "select": {"us": sel_us, "bytes": proj_b + edge_b, "GB/s": (proj_b + edge_b) / sel_us / 1e3,
                   "frac_hbm": (proj_b + edge_b) / sel_us / 1e3 / hbm,
                   "TFLOP/s_project": proj_f / sel_us / 1e6, "plan": plan,
                   "project_then_edges_us": 1000.0 * statistics.median(t_pair)},
        "timing": "median of per-step event intervals; L2 flushed before every step",
    }


def gather_ceiling(w, dev, stream, flush, record_ext, L, steps):
    """Random-row gather rate of this GPU (dflash2_probe_gather), the bound of the
    edge kernel's codebook reads: the workload's gather volume (2 rows of R per
    candidate per transition) read as rows of 128, 256 and 512 bytes at uniform
    random ids from a table the size of the two codebooks, L2 flushed between
    launches."""
    import ctypes

    import torch
    b = 2 if w.dtype == "bf16" else 4
    E = w.S_sel * max(w.n_sel - 1, 0)
    table_bytes = 2 * w.V * w.R * b
    gather_bytes = 2 * E * w.K * w.R * b
    if gather_bytes == 0:
        return None
    g = torch.Generator().manual_seed(4242)
    out = {"table_bytes": table_bytes, "gathered_bytes": gather_bytes,
           "note": "read-only random gathers at uniform ids (4 bytes written per row), one CTA "
                   "per SM with its ids staged on chip and 16-byte cp.async into a shared-memory "
                   "ring: the way the edge kernels read R*b-byte codebook rows"}
    sp = ctypes.c_void_p(stream.cuda_stream)
    f = L.dflash2_probe_gather
    big = torch.zeros(8 * table_bytes // 4, dtype=torch.int32, device=dev)
    for rb in (128, 256, 512):
        res_t = {}
        for mult in (1, 8):  # the step's gather volume, and eight times it from a table 8x larger
            table = big[: mult * table_bytes // 4]
            rows = mult * table_bytes // rb
            n_ids = mult * gather_bytes // rb
            ids = torch.randint(0, rows, (n_ids,), generator=g, dtype=torch.int32).to(dev)
            res = torch.empty((n_ids,), dtype=torch.int32, device=dev)
            args = (ctypes.c_void_p(table.data_ptr()), rows, rb, ctypes.c_void_p(ids.data_ptr()),
                    n_ids, ctypes.c_void_p(res.data_ptr()), sp)
            _call(f, args, L)
            if record_ext is not None:
                t = _timed_graph(steps, stream, flush, [(f, args)], record_ext, L)[0]
            else:
                t = _timed_eager(steps, stream, flush, [(f, args)], L)[0]
            res_t[mult] = (1000.0 * statistics.median(t), n_ids * (rb + 4))
            del ids, res
        (us1, b1), (us8, b8) = res_t[1], res_t[8]
        marginal = (b8 - b1) / (us8 - us1) / 1e3
        out[f"rows_{rb}B"] = {"us": us1, "GB/s": b1 / us1 / 1e3,
                              "frac_hbm": b1 / us1 / 1e3 / _peaks()[0],
                              "us_8x": us8, "marginal_GB/s": marginal,
                              "marginal_frac_hbm": marginal / _peaks()[0]}
    out["marginal"] = ("marginal rate = (8x bytes - 1x bytes) / (8x time - 1x time), the 8x "
                       "volume drawn from a table 8x larger (beyond L2): the cold gather rate "
                       "with the launch and timing-event cost taken out")
    del big
    return out


# ---------------------------------------------------------------- GPU arm

def main():
    args = _args()
    if args.impl == "reference":
        return run_reference(args)
    rank, world, local = _env()
    import ctypes

    import torch
    import torch.distributed as tdist

    import dflash2_draft_head_gb300 as df2
    from dflash2_draft_head_gb300 import synth

    df2.build_library()
    L = df2.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        tdist.init_process_group("nccl", device_id=dev)
    w0 = _workload(args.workload)
    w = rank_workload(w0, rank)

    bt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    ci = synth.conv_inputs(w)
    cb = synth.codebooks(w0)
    si = synth.selector_inputs(w)
    host_in = {"x": ci["x"].to(bt), "hist": ci["hist"].to(bt), "delta": ci["delta"].to(bt),
               "h": si["h"].to(bt), "cand_ids": si["cand_ids"], "unary": si["unary"]}
    d_in = {k: v.to(dev).contiguous() for k, v in host_in.items()}
    base = ci["base"].to(bt).to(dev)
    Wt = cb["W"].to(bt).to(dev)
    A = cb["A"].to(bt).to(dev)
    B = cb["B"].to(bt).to(dev)
    del ci, cb, si
    out = torch.empty((w.S, w.n, w.C), dtype=bt, device=dev)
    P = w.S_sel * w.n_sel
    E = w.S_sel * max(w.n_sel - 1, 0)
    u = torch.empty((P, w.R), dtype=torch.float32, device=dev)
    best_slot = torch.empty((max(E, 1), w.K), dtype=torch.int32, device=dev)
    best_score = torch.empty((max(E, 1), w.K), dtype=torch.float32, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    code = 1 if w.dtype == "bf16" else 0
    vp = ctypes.c_void_p

    def ptr(t):
        return vp(t.data_ptr())

    conv_args = (ptr(d_in["x"]), ptr(d_in["hist"]), ptr(base), ptr(d_in["delta"]), ptr(out),
                 w.S, w.n, w.C, w.T, w.G, code, code, sp)
    proj_args = (ptr(d_in["h"]), ptr(Wt), ptr(u), P, w.d, w.R, code, sp)
    edge_args = (ptr(d_in["cand_ids"]), ptr(u), ptr(A), ptr(B), ptr(d_in["unary"]), w.S_sel,
                 w.n_sel, w.K, w.R, w.V, code, None, ptr(best_slot), ptr(best_score), ptr(flag),
                 sp)
    sel_args = (ptr(d_in["h"]), ptr(Wt), ptr(d_in["cand_ids"]), ptr(A), ptr(B),
                ptr(d_in["unary"]), w.S_sel, w.n_sel, w.d, w.K, w.R, w.V, code, ptr(u), None,
                ptr(best_slot), ptr(best_score), ptr(flag), sp)
    f_conv, f_proj, f_edge = L.dflash2_dynconv, L.dflash2_project, L.dflash2_edges
    f_sel = L.dflash2_select

    def step():
        r = f_conv(*conv_args) | f_sel(*sel_args)
        if r:
            raise RuntimeError(L.dflash2_last_error().decode())

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            tdist.barrier()

    torch.cuda.set_stream(stream)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    barrier()

    K = args.steps
    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    record_ext = None if args.no_graph else _event_record_external()
    timer = _timer(stream, record_ext, L)
    mode = "cuda-graph" if record_ext is not None else "eager"
    calls = [(f_conv, conv_args), (f_sel, sel_args)]
    with ClockSampler(gpu_uuid) as clk:
        barrier()
        wall0 = time.perf_counter()
        # the timed steps: one event before the step's first call, one after its last
        t_step = timer(K, flush, calls, ends_only=True)
        barrier()
        wall = time.perf_counter() - wall0
    K_iso = max(min(K, 200), 1)
    # the same step with an event between the two calls: each call's share
    t_conv, t_sel = timer(K_iso, flush, calls)
    sel_plan = _select_fused(L, w0)
    # each call's device time launched back to back (no event between the calls)
    b2b_conv = _back_to_back_us(stream, flush, [(f_conv, conv_args)], L)
    b2b_sel = _back_to_back_us(stream, flush, [(f_sel, sel_args)], L)
    # the projection and the edge kernel on their own (the path dflash2_select
    # takes for shapes the one-kernel selector does not run)
    iso_calls = [(f_proj, proj_args), (f_edge, edge_args)]
    if record_ext is not None:
        t_proj, t_edge = _timed_graph(K_iso, stream, flush, iso_calls, record_ext, L)
        # the projection again with h left in L2 ("warm": no flush between launches)
        t_proj_warm = _timed_graph(K_iso, stream, _NoFlush(), [(f_proj, proj_args)], record_ext,
                                   L)[0]
    else:
        t_proj, t_edge = _timed_eager(K_iso, stream, flush, iso_calls, L)
        t_proj_warm = _timed_eager(K_iso, stream, _NoFlush(), [(f_proj, proj_args)], L)[0]
    # top-K candidate extraction, the step before the selector, on the draft
    # logits of the same positions: [P, V] fp32 rows (the review thread's
    # top-k microbenchmark runs fp32 rows); also an isolated loop
    logits = synth.logits_rows(w.seed, 0, P, w.V, "f32").to(dev)
    tk_ids = torch.empty((P, w.K), dtype=torch.int32, device=dev)
    tk_vals = torch.empty((P, w.K), dtype=torch.float32, device=dev)
    topk_args = (ptr(logits), P, w.V, w.K, 0, ptr(tk_ids), ptr(tk_vals), sp)
    f_topk = L.dflash2_topk
    _call(f_topk, topk_args, L)  # first call per device queries occupancy (not capturable)
    barrier()
    if record_ext is not None:
        t_topk = _timed_graph(K_iso, stream, flush, [(f_topk, topk_args)], record_ext, L)[0]
    else:
        t_topk = _timed_eager(K_iso, stream, flush, [(f_topk, topk_args)], L)[0]
    topk_b = P * w.V * 4 + P * w.K * 8
    topk_us = 1000.0 * statistics.mean(t_topk)
    # the same extraction for one draft block (one sequence's n rows): the decode
    # case, latency-bound; fp32 and bf16 rows
    blk = {}
    for lname, lt in (("f32", logits[:w.n]), ("bf16", logits[:w.n].to(torch.bfloat16))):
        lt = lt.contiguous()
        b_args = (ptr(lt), w.n, w.V, w.K, 1 if lname == "bf16" else 0, ptr(tk_ids), ptr(tk_vals),
                  sp)
        _call(f_topk, b_args, L)
        if record_ext is not None:
            tb = _timed_graph(K_iso, stream, flush, [(f_topk, b_args)], record_ext, L)[0]
        else:
            tb = _timed_eager(K_iso, stream, flush, [(f_topk, b_args)], L)[0]
        bb = w.n * w.V * (2 if lname == "bf16" else 4) + w.n * w.K * 8
        bu = 1000.0 * statistics.mean(tb)
        blk[lname] = {"us": bu, "bytes": bb, "GB/s": bb / bu / 1e3,
                      "frac_hbm": bb / bu / 1e3 / _peaks()[0]}
        del lt
    del logits
    # delta predictor (delta = x . Wc^T, the conv's taps from its input), bf16 on
    # the tensor cores; the conv inputs of the step
    TG = w.T * w.G
    Wc = synth.conv_proj(w0).to(bt).to(dev)
    d_pred = torch.empty((w.S, w.n, w.T, w.G), dtype=bt, device=dev)
    pd_args = (ptr(d_in["x"]), ptr(Wc), ptr(d_pred), w.S * w.n, w.C, TG, code, sp)
    f_pd = L.dflash2_predict_delta
    _call(f_pd, pd_args, L)
    if record_ext is not None:
        t_pd = _timed_graph(K_iso, stream, flush, [(f_pd, pd_args)], record_ext, L)[0]
    else:
        t_pd = _timed_eager(K_iso, stream, flush, [(f_pd, pd_args)], L)[0]
    pd_us = 1000.0 * statistics.mean(t_pd)
    bsz = 2 if w.dtype == "bf16" else 4
    pd_b = (w.S * w.n * w.C + TG * w.C + w.S * w.n * TG) * bsz
    pd_f = 2.0 * w.S * w.n * w.C * TG
    # the conv with its taps predicted inside the kernel (delta never leaves the
    # chip, x read from HBM once), against the unfused pair it replaces: predict,
    # then convolve the stored delta, on the same inputs and output buffer
    fz = None
    if w.dtype == "bf16" and TG <= 256 and TG % 8 == 0 and w.T <= 8:
        f_fz = L.dflash2_dynconv_predicted
        fz_args = (ptr(d_in["x"]), ptr(d_in["hist"]), ptr(base), ptr(Wc), ptr(out), w.S, w.n,
                   w.C, w.T, w.G, code, code, sp)
        pair_conv = (ptr(d_in["x"]), ptr(d_in["hist"]), ptr(base), ptr(d_pred), ptr(out), w.S,
                     w.n, w.C, w.T, w.G, code, code, sp)
        _call(f_fz, fz_args, L)
        if record_ext is not None:
            t_fz = _timed_graph(K_iso, stream, flush, [(f_fz, fz_args)], record_ext, L)[0]
            t_pair = _timed_graph(K_iso, stream, flush, [(f_pd, pd_args), (f_conv, pair_conv)],
                                  record_ext, L)
        else:
            t_fz = _timed_eager(K_iso, stream, flush, [(f_fz, fz_args)], L)[0]
            t_pair = _timed_eager(K_iso, stream, flush, [(f_pd, pd_args), (f_conv, pair_conv)], L)
        fz_us = 1000.0 * statistics.mean(t_fz)
        pair_us = 1000.0 * statistics.mean(a + b for a, b in zip(t_pair[0], t_pair[1]))
        # algorithmic bytes: x, history, base taps and Wc read once, out written once
        fz_b = (2 * w.S * w.n * w.C + w.S * (w.T - 1) * w.C + w.T * w.C + TG * w.C) * bsz
        fz = {"isolated": True, "steps": K_iso, "us": fz_us, "bytes": fz_b,
              "GB/s": fz_b / fz_us / 1e3, "frac_hbm": fz_b / fz_us / 1e3 / _peaks()[0],
              "TFLOP/s": pd_f / fz_us / 1e6, "unfused_pair_us": pair_us,
              "speedup_vs_pair": pair_us / fz_us,
              "note": "delta = x . Wc^T and the conv in one kernel; not part of the timed step "
                      "(its conv takes delta as an input)"}
    del Wc, d_pred
    # greedy chain readout (p_min cut) after the selector: the edge scores of the
    # same step materialised once (outside timing), then an isolated loop
    e_full = torch.empty((max(E, 1), w.K, w.K), dtype=torch.float32, device=dev)
    _call(f_edge, edge_args[:11] + (ptr(e_full),) + edge_args[12:], L)
    ch_tok = torch.empty((w.S_sel, w.n_sel), dtype=torch.int32, device=dev)
    ch_pr = torch.empty((w.S_sel, w.n_sel), dtype=torch.float32, device=dev)
    ch_len = torch.empty((w.S_sel,), dtype=torch.int32, device=dev)
    chain_args = (ptr(d_in["cand_ids"]), ptr(d_in["unary"]), ptr(e_full), ptr(best_slot), None,
                  w.S_sel, w.n_sel, w.K, ctypes.c_float(P_MIN), ptr(ch_tok), ptr(ch_pr),
                  ptr(ch_len), ptr(flag), sp)
    f_chain = L.dflash2_chain
    if record_ext is not None:
        t_chain = _timed_graph(K_iso, stream, flush, [(f_chain, chain_args)], record_ext, L)[0]
    else:
        t_chain = _timed_eager(K_iso, stream, flush, [(f_chain, chain_args)], L)[0]
    chain_us = 1000.0 * statistics.mean(t_chain)
    # bytes: argmax table, the n-1 chosen edge rows, the unary row, the chosen ids
    # (one 4-byte word each) and the outputs, per sequence
    chain_b = w.S_sel * (2 * max(w.n_sel - 1, 0) * w.K * 4 + w.K * 4 + w.n_sel * 4
                         + w.n_sel * 8 + 4)
    del e_full
    gather = gather_ceiling(w, dev, stream, flush, record_ext, L, K_iso)
    # the other workloads' steps (rank 0 of a single-GPU run)
    workloads = {}
    if world == 1 and not args.no_workloads:
        from dflash2_draft_head_gb300.workloads import WORKLOADS
        for wk in WORKLOADS:
            if wk.name != w0.name:
                workloads[wk.name] = workload_leg(wk.name, dev, stream, flush, timer, L,
                                                  K_iso)
                torch.cuda.empty_cache()
    total_ms = max_over_ranks(sum(t_step), world, dev)
    if int(flag.item()) != 0 or df2.take_device_faults() != 0:
        raise RuntimeError("device error flag set during the benchmark")

    # end to end through the public API: pinned host inputs -> device -> readout -> host
    pin = {k: v.pin_memory() for k, v in host_in.items()}
    h_slot = torch.empty(best_slot.shape, dtype=torch.int32).pin_memory()
    h_score = torch.empty(best_score.shape, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = h_slot.numel() * 4 + h_score.numel() * 4

    # Two device input sets: step k+1's host->device copies (two copy streams, the
    # tensors split between them) overlap step k's kernels; every step still copies
    # its inputs in and its readout out inside the timed region.
    d_in2 = {k2: torch.empty_like(v) for k2, v in d_in.items()}
    sets = [d_in, d_in2]

    def step_args(di):
        ca = (ptr(di["x"]), ptr(di["hist"]), ptr(base), ptr(di["delta"]), ptr(out),
              w.S, w.n, w.C, w.T, w.G, code, code, sp)
        sa = (ptr(di["h"]), ptr(Wt), ptr(di["cand_ids"]), ptr(A), ptr(B), ptr(di["unary"]),
              w.S_sel, w.n_sel, w.d, w.K, w.R, w.V, code, ptr(u), None, ptr(best_slot),
              ptr(best_score), ptr(flag), sp)
        return ca, sa

    args2 = [step_args(di) for di in sets]
    copy_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    names = sorted(pin, key=lambda k2: -pin[k2].numel() * pin[k2].element_size())
    split = [names[0::2], names[1::2]]  # largest tensors alternate between the streams
    ready = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]  # [set][copy stream]
    free = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(k):
        b = k % 2
        for j, cst in enumerate(copy_streams):
            if used[b]:
                cst.wait_event(free[b])  # the kernels that read this set are done
            with torch.cuda.stream(cst):
                for k2 in split[j]:
                    sets[b][k2].copy_(pin[k2], non_blocking=True)
            ready[b][j].record(cst)
        for j in range(2):
            stream.wait_event(ready[b][j])
        ca, sa = args2[b]
        r = f_conv(*ca) | f_sel(*sa)
        if r:
            raise RuntimeError(L.dflash2_last_error().decode())
        free[b].record(stream)
        used[b] = True
        h_slot.copy_(best_slot, non_blocking=True)
        h_score.copy_(best_score, non_blocking=True)

    for k in range(3):
        e2e_step(k)
    barrier()
    E2 = max(args.e2e_steps, 1)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for cst in copy_streams:
        cst.wait_event(e0)  # no copy of the timed steps starts before the start event
    for k in range(E2):
        e2e_step(k)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    link = _host_link(pin, d_in, copy_streams, split, stream)

    positions = w.S * w.n * world
    value = positions * K / (total_ms / 1000.0)
    conv_b, proj_b, proj_f, edge_b = _bytes(w)
    hbm, tc, src = _peaks()
    conv_us = 1000.0 * statistics.mean(t_conv)
    sel_us = 1000.0 * statistics.mean(t_sel)
    proj_us = 1000.0 * statistics.mean(t_proj)
    edge_us = 1000.0 * statistics.mean(t_edge)

    def _traffic(kernel, fname):
        sha = hashlib.sha256(open(os.path.join(ROOT, "dflash2_draft_head_gb300", "csrc", fname),
                                  "rb").read()).hexdigest()
        tr = TRAFFIC.get((w.name, kernel))
        return tr["bytes"] if tr and tr["sha"] == sha else None
    # the dominant kernel of the step: the call with the larger share of its time
    if sel_us >= conv_us:
        dom = {"kernel": "dflash2_select" + ("" if sel_plan["fused"] else " (project + edges)"),
               "bytes": proj_b + edge_b, "us": sel_us,
               "traffic": _traffic("select", "select.cu") if sel_plan["fused"] else None,
               "b2b": b2b_sel}
    else:
        dom = {"kernel": "dflash2_dynconv", "bytes": conv_b, "us": conv_us,
               "traffic": _traffic("dynconv", "dynconv.cu"), "b2b": b2b_conv}
    achieved = dom["bytes"] / (dom["us"] * 1e-6) / 1e9
    traffic = _traffic("dynconv", "dynconv.cu")
    tk_sha = hashlib.sha256(open(os.path.join(ROOT, "dflash2_draft_head_gb300", "csrc",
                                              "topk.cu"), "rb").read()).hexdigest()
    tr = TRAFFIC.get((w.name, "topk"))
    topk_traffic = tr["bytes"] if tr and tr["sha"] == tk_sha else None
    fz_sha = hashlib.sha256(open(os.path.join(ROOT, "dflash2_draft_head_gb300", "csrc",
                                              "dynconv_pred.cu"), "rb").read()).hexdigest()
    tr = TRAFFIC.get((w.name, "dynconv_predicted"))
    fz_traffic = tr["bytes"] if tr and tr["sha"] == fz_sha else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": _config(w0, world),
        "roofline": {"bound": "hbm", "kernel": dom["kernel"], "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": dom["traffic"], "bytes_per_launch": dom["bytes"],
                     "us_per_launch": dom["us"], "peak_source": src,
                     "timing": "live, an event between the step's two calls",
                     "back_to_back_us": dom["b2b"],
                     "frac_back_to_back": dom["bytes"] / dom["b2b"] / 1e3 / hbm},
        "roofline_step": {"bound": "hbm", "bytes_per_step": conv_b + proj_b + edge_b,
                          "us_per_step": 1000.0 * total_ms / K,
                          "achieved": (conv_b + proj_b + edge_b) / (1000.0 * total_ms / K) / 1e3,
                          "peak": hbm, "unit": "GB/s",
                          "frac": (conv_b + proj_b + edge_b) / (1000.0 * total_ms / K) / 1e3 / hbm},
        "roofline_all": {
            "dynconv": {"bound": "hbm", "achieved": conv_b / conv_us / 1e3, "peak": hbm,
                        "unit": "GB/s", "frac": conv_b / conv_us / 1e3 / hbm,
                        "traffic": traffic},
            "select": {"bound": "hbm", "achieved": (proj_b + edge_b) / sel_us / 1e3, "peak": hbm,
                       "unit": "GB/s", "frac": (proj_b + edge_b) / sel_us / 1e3 / hbm,
                       "traffic": dom["traffic"] if dom["kernel"] == "dflash2_select" else
                       (_traffic("select", "select.cu") if sel_plan["fused"] else None),
                       "plan": sel_plan},
            "project": {"bound": "hbm", "achieved": proj_b / proj_us / 1e3, "peak": hbm,
                        "unit": "GB/s", "frac": proj_b / proj_us / 1e3 / hbm,
                        "tensor_TFLOP/s": proj_f / proj_us / 1e6, "tensor_peak": tc,
                        "tensor_frac": proj_f / proj_us / 1e6 / tc, "timing": "isolated loop"},
            "edges": {"bound": "hbm", "achieved": edge_b / edge_us / 1e3, "peak": hbm,
                      "unit": "GB/s", "frac": edge_b / edge_us / 1e3 / hbm,
                      "timing": "isolated loop"},
            "topk": {"bound": "hbm", "achieved": topk_b / topk_us / 1e3, "peak": hbm,
                     "unit": "GB/s", "frac": topk_b / topk_us / 1e3 / hbm,
                     "traffic": topk_traffic, "timing": "isolated loop"},
            "dynconv_predicted": None if fz is None else {
                "bound": "hbm", "achieved": fz["bytes"] / fz["us"] / 1e3, "peak": hbm,
                "unit": "GB/s", "frac": fz["bytes"] / fz["us"] / 1e3 / hbm,
                "traffic": fz_traffic, "timing": "isolated loop"},
        },
        "kernels": {
            "dynconv": {"us": conv_us, "bytes": conv_b, "GB/s": conv_b / conv_us / 1e3,
                        "frac_hbm": conv_b / conv_us / 1e3 / hbm,
                        "back_to_back_us": b2b_conv,
                        "frac_hbm_back_to_back": conv_b / b2b_conv / 1e3 / hbm,
                        "positions_per_s": positions / (conv_us * 1e-6)},
            "select": {"us": sel_us, "bytes": proj_b + edge_b,
                       "GB/s": (proj_b + edge_b) / sel_us / 1e3,
                       "frac_hbm": (proj_b + edge_b) / sel_us / 1e3 / hbm,
                       "back_to_back_us": b2b_sel,
                       "frac_hbm_back_to_back": (proj_b + edge_b) / b2b_sel / 1e3 / hbm,
                       "plan": sel_plan,
                       "note": "dflash2_select in the step (one kernel when plan.fused)"},
            "project": {"isolated": True, "steps": K_iso, "us": proj_us, "bytes": proj_b,
                        "warm_us": 1000.0 * statistics.mean(t_proj_warm),
                        "GB/s": proj_b / proj_us / 1e3,
                        "TFLOP/s": proj_f / proj_us / 1e6,
                        "frac_hbm": proj_b / proj_us / 1e3 / hbm,
                        "frac_bf16_tc": proj_f / proj_us / 1e6 / tc},
            "edges": {"isolated": True, "steps": K_iso, "us": edge_us, "bytes": edge_b,
                      "GB/s": edge_b / edge_us / 1e3,
                      "frac_hbm": edge_b / edge_us / 1e3 / hbm},
            "predict_delta": {"isolated": True, "steps": K_iso, "us": pd_us, "bytes": pd_b,
                              "TFLOP/s": pd_f / pd_us / 1e6, "GB/s": pd_b / pd_us / 1e3,
                              "frac_hbm": pd_b / pd_us / 1e3 / hbm,
                              "frac_bf16_tc": pd_f / pd_us / 1e6 / tc,
                              "note": "delta = x . Wc^T (C -> T*G), unfused, before the conv"},
            "dynconv_predicted": fz,
            "chain": {"isolated": True, "steps": K_iso, "us": chain_us, "bytes": chain_b,
                      "p_min": P_MIN, "GB/s": chain_b / chain_us / 1e3,
                      "bound": "latency (a walk of n dependent lookups per sequence)",
                      "note": "not part of the timed step; readout after it"},
            "topk": {"isolated": True, "steps": K_iso, "us": topk_us, "bytes": topk_b,
                     "rows": P, "V": w.V, "K": w.K, "logits": "f32",
                     "GB/s": topk_b / topk_us / 1e3, "frac_hbm": topk_b / topk_us / 1e3 / hbm,
                     "note": "not part of the timed step; candidate extraction before it"},
            "topk_draft_block": {"isolated": True, "steps": K_iso, "rows": w.n, "V": w.V,
                                 "K": w.K, **blk,
                                 "note": "one sequence's draft block (the decode case)"},
        },
        "gather_ceiling": gather,
        "workloads": workloads,
        "e2e": {"value": positions * E2 / (e2e_ms / 1000.0), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E2,
                "pipelining": "double-buffered inputs: step k+1's H2D copies (2 streams) overlap "
                              "step k's kernels",
                # the host link alone: one step's inputs copied with no kernel running
                "host_link": {**link,
                              "bound_positions_per_s": positions / (
                                  h2d / (1e9 * max(link["GB/s_1stream"], link["GB/s_2streams"]))),
                              "frac_of_bound": (positions * E2 / (e2e_ms / 1000.0)) / (
                                  positions / (h2d / (1e9 * max(link["GB/s_1stream"],
                                                                link["GB/s_2streams"]))))}},
        # dynconv + the selector (one kernel, or project + edges) per timed step
        "gpu_launches": (2 if sel_plan["fused"] else 3) * K,
        "clocks": clk.summary(),
        "torch": torch.__version__,
        "inputs_sha256": _input_digests(host_in),
        "wall_s_timed_region": wall,
        "launch_mode": mode,
        "cpu_baseline": None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w0, args.cpu_seconds)
    if world > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
