"""Benchmark of the MoE routing path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the routing hot path over one batch of synthetic
router logits, T=8192 tokens x E=2304 experts, topk=36, fp32, softmax:
router forward (probs, routing_map, intermediate, topk_idx, topk_w), router
backward, aux-loss scores forward and aux-loss scores backward -- the four
kernels TransformerEngine PR 3012 reports effective bandwidth for. The metric
is effective GB/s: the minimum bytes each kernel must move (the page's rule:
fwd reads logits and writes probs, routing_map and intermediate) over device
time. Prints ONE JSON line (rank 0).

Also reported in the same line: per-kernel GB/s on the other large-T
workloads, fused decode route+sort in us/call (eager and CUDA-graph replayed,
against the launch floor), the prefill route+sort, the end-to-end rate through
host buffers, the roofline of the dominant kernel and the CPU oracle baseline.

--impl reference times the CPU oracle (the reference implementation here) on a
bounded sample of the same workload and prints the same line shape.

Multi-GPU: one process per GPU (torchrun); every rank routes its own T=8192
batch (tokens are independent, so there is no collective on the data path);
value = bytes of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "effective GB/s vs 8 TB/s HBM (T=8192); µs/call fused route+sort at T≤16"
WORKLOAD = "router fwd+bwd+aux fwd+aux bwd, T=8192 E=2304 topk=36 fp32 softmax"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "router_fwd_T8192_E2304_k36.md")
PAGE_B300 = {  # TransformerEngine PR 3012 "Performance" (B300 SXM6, fp32, T=8192), context only
    ("fwd", "softmax", 2304, 36): 964, ("bwd", "softmax", 2304, 36): 2766,
    ("aux_fwd", "softmax", 2304, 36): 891, ("aux_bwd", "softmax", 2304, 36): 4201,
    ("fwd", "softmax", 512, 4): 1784, ("fwd", "softmax", 512, 8): 904, ("fwd", "softmax", 512, 22): 924,
    ("fwd", "softmax", 512, 36): 908, ("bwd", "softmax", 512, 22): 5362, ("aux_fwd", "softmax", 512, 22): 896,
    ("aux_bwd", "softmax", 512, 22): 6155, ("fwd", "sigmoid", 2304, 36): 798, ("bwd", "sigmoid", 2304, 36): 2274,
    ("aux_fwd", "sigmoid", 2304, 36): 867, ("aux_bwd", "sigmoid", 2304, 36): 2757,
}


def kernel_bytes(kind: str, T: int, E: int, topk: int, in_bytes: int = 4, compact: bool = True) -> int:
    """Algorithmic bytes of one launch (page-3 rule; compact outputs added when written)."""
    n = T * E
    if kind == "fwd":
        b = n * (in_bytes + in_bytes + 1 + 4)
        return b + (T * topk * 8 if compact else 0)
    if kind == "bwd":
        return n * (4 + 4 + 1 + 4)
    if kind == "aux_fwd":
        return n * (in_bytes + 4 + 1)
    if kind == "aux_bwd":
        return n * (4 + 4 + 4)
    raise ValueError(kind)


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# the sources the wide forward kernel is compiled from (its traffic figure is
# void once any of them changes)
FWD_SOURCES = ("common.cuh", "route.cuh", "route_wide.cuh", "internal.h", "fwd.cu")


def _code_only(text: str) -> str:
    """The source with its comments and blank lines taken out, so that the hash
    follows the code a profile was taken on, not its commentary."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_gating_expert_row_gb300", "csrc")
    for f in FWD_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    if it was taken on the current kernel sources (else None)."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    text = open(PROFILE_TRAFFIC).read()
    src = traf = None
    for line in text.splitlines():
        if line.startswith("kernel_source_hash:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traf = int(line.split(":", 1)[1].strip())
    if src != kernel_source_hash():
        return None
    return traf


# ---------------------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (ts, l) in self.lines if t0 - 0.05 <= ts <= t1 + 0.05] or [l for _, l in self.lines[-3:]]
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------------------- ours


class Timer:
    """Per-kernel CUDA events on the launching stream."""

    def __init__(self, stream):
        self.stream = stream
        self.pairs = {}

    def around(self, name, fn):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        fn()
        b.record(self.stream)
        self.pairs.setdefault(name, []).append((a, b))

    def mean_ms(self, name):
        ps = self.pairs.get(name, [])
        return sum(a.elapsed_time(b) for a, b in ps) / max(1, len(ps))


def make_step(mr, w, dev, stream):
    """Allocates the step's tensors and returns the list of (name, launch) pairs."""
    T, E, k = w.T, w.E, w.topk
    x = w.make_logits().to(dev)
    g = synth.grad(T, E).to(dev)
    b = w.make_bias()
    b = b.to(dev) if b is not None else None
    f32 = dict(dtype=torch.float32, device=dev)
    t = dict(x=x, g=g, bias=b, probs=torch.empty(T, E, dtype=x.dtype, device=dev),
             map=torch.empty(T, E, dtype=torch.uint8, device=dev), inter=torch.empty(T, E, **f32),
             idx=torch.empty(T, k, dtype=torch.int32, device=dev), w=torch.empty(T, k, **f32),
             dx=torch.empty(T, E, **f32), scores=torch.empty(T, E, **f32),
             amap=torch.empty(T, E, dtype=torch.uint8, device=dev), adx=torch.empty(T, E, **f32))
    p = mr.RouterParams(T=T, E=E, topk=k, score_fn=w.score_fn, in_dtype=w.in_dtype, renorm=w.renorm,
                        scaling=w.scaling, bias=b)
    cp = p.c()
    L = mr._lib
    s = stream.cuda_stream
    P = ctypes.byref(cp)
    ptr = {n: (v.data_ptr() if v is not None else None) for n, v in t.items()}

    # The launches pass raw device pointers, so they must keep the tensors (and
    # the params, which hold the bias) alive: every launch goes through chk,
    # whose default argument holds them for as long as any launch exists.
    def chk(rc, what, _owned=(t, p, cp)):
        if rc != 0:
            raise RuntimeError(f"{what}: {mr.strerror(rc)}")

    launches = [
        ("fwd", lambda: chk(L.moe_router_fwd(P, ptr["x"], ptr["probs"], ptr["map"], ptr["inter"], ptr["idx"],
                                             ptr["w"], None, s), "fwd")),
        ("bwd", lambda: chk(L.moe_router_bwd(P, ptr["g"], ptr["inter"], ptr["map"], ptr["dx"], s), "bwd")),
        ("aux_fwd", lambda: chk(L.moe_aux_scores_fwd(T, E, k, w.score_fn, w.in_dtype, ptr["x"], ptr["scores"],
                                                     ptr["amap"], s), "aux_fwd")),
        ("aux_bwd", lambda: chk(L.moe_aux_scores_bwd(T, E, w.score_fn, ptr["g"], ptr["scores"], ptr["adx"], s),
                                "aux_bwd")),
    ]
    return launches, t, p


def step_bytes(w, kinds=("fwd", "bwd", "aux_fwd", "aux_bwd")) -> dict:
    ib = 2 if w.in_dtype == synth.BF16 else 4
    return {kd: kernel_bytes(kd, w.T, w.E, w.topk, ib) for kd in kinds}


def time_kernels(mr, w, dev, stream, calls=20, replays=5) -> dict:
    """Per-kernel device time of one workload's step kernels. A kernel of these
    sizes runs for tens of µs, about as long as a Python launch, so each kernel
    is timed as a CUDA-graph replay of `calls` back-to-back calls that rotate
    over enough buffer sets (more than 3x L2 in all) that every call reads its
    inputs from HBM."""
    per_set = None
    sets = []
    while not sets or len(sets) * per_set < 3 * 129 * 2 ** 20 or len(sets) < 2:
        launches, t, _ = make_step(mr, w, dev, stream)
        per_set = sum(v.numel() * v.element_size() for v in t.values() if v is not None)
        with torch.cuda.stream(stream):
            for _, fn in launches:  # valid bwd / aux inputs in every set
                fn()
        sets.append(dict(launches))  # each launch owns its set's tensors (see make_step)
    torch.cuda.synchronize()
    out = {}
    fn_name = "softmax" if w.score_fn == synth.SOFTMAX else "sigmoid"
    for name, nb in step_bytes(w).items():
        it = iter(range(10 ** 9))
        with plain_order(mr):
            us = graph_us(lambda: sets[next(it) % len(sets)][name](), stream, calls, replays)
        gbs = nb / (us * 1e-6) / 1e9
        d = {"us": round(us, 2), "GB/s": round(gbs, 1)}
        page = PAGE_B300.get((name, fn_name, w.E, w.topk))
        if page:
            d["page_B300_GB/s"] = page
        out[name] = d
    out["timing"] = f"CUDA graph, {calls} calls per replay over {len(sets)} buffer sets ({len(sets) * per_set >> 20} MB)"
    return out


def bf16_rates(mr, dev, stream, calls=20, replays=5) -> dict:
    """The headline shape with bf16 logits: T=8192 E=2304 topk=36 softmax; the forward
    writes bf16 probs, the backward takes and returns bf16 gradients (the
    intermediate stays fp32): 9 bytes per element each. Graph replays rotating
    over buffer sets larger than 3x L2."""
    w = synth.Workload("softmax_T8192_E2304_k36_bf16", 8192, 2304, 36, synth.SOFTMAX, synth.BF16)
    sets = []
    while len(sets) < 3:
        launches, t, p = make_step(mr, w, dev, stream)
        g16 = t["g"].to(torch.bfloat16)
        dx16 = torch.empty_like(g16)
        cp = p.c()
        L, s = mr._lib, stream.cuda_stream

        def bwd(cp=cp, g16=g16, dx16=dx16, t=t, owned=(p, launches)):
            rc = L.moe_router_bwd_dtype(ctypes.byref(cp), mr.MR_BF16, g16.data_ptr(), t["inter"].data_ptr(),
                                        t["map"].data_ptr(), dx16.data_ptr(), s)
            if rc != 0:
                raise RuntimeError(mr.strerror(rc))

        with torch.cuda.stream(stream):
            dict(launches)["fwd"]()
        sets.append({"fwd": dict(launches)["fwd"], "bwd_bf16": bwd})
    torch.cuda.synchronize()
    n = w.T * w.E
    nbytes = {"fwd": kernel_bytes("fwd", w.T, w.E, w.topk, 2), "bwd_bf16": n * (2 + 4 + 1 + 2)}
    pk = peaks()["hbm_gbs"]
    out = {"workload": w.name, "timing": f"CUDA graph, {calls} calls per replay over {len(sets)} buffer sets"}
    for name, nb in nbytes.items():
        it = iter(range(10 ** 9))
        with plain_order(mr):
            us = graph_us(lambda: sets[next(it) % len(sets)][name](), stream, calls, replays)
        gbs = nb / (us * 1e-6) / 1e9
        out[name] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / pk, 3)}
    return out


def decode_latency(mr, dev, stream, n_calls=200, Ts=synth.DECODE_BENCH_TS, shape=synth.decode) -> dict:
    """Fused vs unfused decode route+sort (default E=256, topk=8, bf16), eager and graph."""
    L = mr._lib
    res = {}
    s = stream.cuda_stream

    def checked(fn):
        def run(st):
            rc = fn(st)
            if rc != 0:
                raise RuntimeError(f"decode call failed: {mr.strerror(rc)}")
        return run

    def eager(fn):
        fn = checked(fn)
        with torch.cuda.stream(stream):
            for _ in range(20):
                fn(s)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(n_calls):
                fn(s)
            torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n_calls * 1e6

    def graph(fn):
        fn = checked(fn)
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(cs):
            for _ in range(5):
                fn(cs.cuda_stream)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(n_calls):
                fn(cs.cuda_stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        reps = 10
        with torch.cuda.stream(cs):  # replay() launches on the current stream
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            a.record(cs)
            for _ in range(reps):
                g.replay()
            b.record(cs)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * n_calls)

    noop = lambda st: L.moe_router_noop(st)  # noqa: E731
    floor = {"eager_us": round(eager(noop), 2), "graph_us": round(graph(noop), 2)}
    mr.moe_router_set_launch_overlap(False)
    try:
        floor["graph_plain_us"] = round(graph(noop), 2)
    finally:
        mr.moe_router_set_launch_overlap(True)
    res["launch_floor"] = floor
    for T in Ts:
        w = shape(T)
        x = w.make_logits().to(dev)
        p = mr.RouterParams(T=T, E=w.E, topk=w.topk, in_dtype=w.in_dtype, renorm=w.renorm)
        cp = p.c()
        P = ctypes.byref(cp)
        bufs = mr.sort_buffers(T, w.topk, w.E, w.block_m, dev)
        idx = torch.empty(T, w.topk, dtype=torch.int32, device=dev)
        wt = torch.empty(T, w.topk, dtype=torch.float32, device=dev)
        ws = torch.empty(mr.moe_sort_workspace_bytes(T, w.topk, w.E, w.block_m), dtype=torch.uint8, device=dev)
        a = [bufs[n].data_ptr() for n in ("sorted_token_ids", "sorted_weights", "expert_ids", "num_tokens_post_pad")]
        xp, ip, wp, wsp, wsn = x.data_ptr(), idx.data_ptr(), wt.data_ptr(), ws.data_ptr(), ws.numel()

        def fused(st):
            return L.moe_router_fused_fwd_sort(P, xp, w.block_m, ip, wp, a[0], a[1], a[2], a[3], None, 0, None, st)

        def unfused(st):
            L.moe_router_fwd(P, xp, None, None, None, ip, wp, None, st)
            return L.moe_sort(ip, wp, T, w.topk, w.E, w.block_m, a[0], a[1], a[2], a[3], wsp, wsn, None, st)

        fe, fg = eager(fused), graph(fused)
        ue, ug = eager(unfused), graph(unfused)
        # the same calls launched in plain stream order (no launch overlap)
        mr.moe_router_set_launch_overlap(False)
        try:
            fgp, ugp = graph(fused), graph(unfused)
        finally:
            mr.moe_router_set_launch_overlap(True)
        res[f"T={T}"] = {"fused_eager_us": round(fe, 2), "fused_graph_us": round(fg, 2),
                         "unfused_eager_us": round(ue, 2), "unfused_graph_us": round(ug, 2),
                         "fused_graph_plain_us": round(fgp, 2), "unfused_graph_plain_us": round(ugp, 2),
                         "fused_graph_minus_floor_us": round(fg - floor["graph_us"], 2),
                         "fused_eager_minus_floor_us": round(fe - floor["eager_us"], 2)}
    res["note"] = ("graph_us: CUDA-graph replays with the launch overlap on (each call may start while the one "
                   "before it finishes); graph_plain_us: plain stream order; the floor is the empty kernel "
                   "launched the same way")
    return res


class plain_order:
    """Within this block the library launches in plain stream order (no launch
    overlap), so back-to-back calls of one kernel are timed one after another."""

    def __init__(self, mr):
        self.mr = mr

    def __enter__(self):
        self.mr.moe_router_set_launch_overlap(False)

    def __exit__(self, *exc):
        self.mr.moe_router_set_launch_overlap(True)


def graph_us(fn, stream, calls=20, replays=5) -> float:
    """Mean device time of fn() in µs: `calls` back-to-back calls captured into a
    CUDA graph on `stream`, replayed `replays` times between two events."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        g.replay()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(replays):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (calls * replays)


def prefill_route_sort(mr, dev, stream, reps=20) -> dict:
    """T=16384, E=384+1 shared, topk=9, bf16 sigmoid + bias, 8 groups keep 4, block_m=64."""
    w = synth.prefill_grouped()
    x = w.make_logits().to(dev)
    b = w.make_bias().to(dev)
    p = mr.RouterParams(T=w.T, E=w.E, topk=w.topk, score_fn=w.score_fn, in_dtype=w.in_dtype, renorm=w.renorm,
                        n_group=w.n_group, topk_group=w.topk_group, n_shared=w.n_shared, scaling=w.scaling,
                        shared_weight=w.shared_weight, bias=b)
    cp = p.c()
    P = ctypes.byref(cp)
    L = mr._lib
    idx = torch.empty(w.T, w.topk, dtype=torch.int32, device=dev)
    wt = torch.empty(w.T, w.topk, dtype=torch.float32, device=dev)
    bufs = mr.sort_buffers(w.T, w.topk, w.E_tot, w.block_m, dev)
    ws = torch.empty(mr.moe_sort_workspace_bytes(w.T, w.topk, w.E_tot, w.block_m), dtype=torch.uint8, device=dev)
    a = [bufs[n].data_ptr() for n in ("sorted_token_ids", "sorted_weights", "expert_ids", "num_tokens_post_pad")]
    s = stream.cuda_stream
    route = lambda: L.moe_router_fwd(P, x.data_ptr(), None, None, None, idx.data_ptr(), wt.data_ptr(), None, s)  # noqa
    srt = lambda: L.moe_sort(idx.data_ptr(), wt.data_ptr(), w.T, w.topk, w.E_tot, w.block_m, a[0], a[1], a[2],  # noqa
                             a[3], ws.data_ptr(), ws.numel(), None, s)
    with torch.cuda.stream(stream):
        for _ in range(3):
            route()
            srt()
    torch.cuda.synchronize()
    fws = torch.empty(max(1, mr.moe_router_fused_workspace_bytes(cp, w.block_m)), dtype=torch.uint8, device=dev)
    fused = lambda: L.moe_router_fused_fwd_sort(P, x.data_ptr(), w.block_m, idx.data_ptr(), wt.data_ptr(), a[0],  # noqa
                                                a[1], a[2], a[3], fws.data_ptr(), fws.numel(), None, s)
    with torch.cuda.stream(stream):
        for _ in range(3):
            if fused() != 0:
                raise RuntimeError("fused prefill call failed")
    torch.cuda.synchronize()
    # tens of µs per call, close to the cost of a Python launch: timed as CUDA-graph replays
    r_us = graph_us(route, stream, reps)
    s_us = graph_us(srt, stream, reps)
    f_us = graph_us(fused, stream, reps)
    with plain_order(mr):
        f_plain = graph_us(fused, stream, reps)
    rb = w.T * w.E * 2 + w.T * w.topk * 8 + w.E * 4
    npp = int(bufs["num_tokens_post_pad"].item())
    sb = w.T * w.topk * 8 + npp * 8 + (npp // w.block_m) * 4 + 4
    return {"workload": w.name, "route_us": round(r_us, 2), "sort_us": round(s_us, 2),
            "route_GB/s": round(rb / (r_us * 1e-6) / 1e9, 1), "sort_GB/s": round(sb / (s_us * 1e-6) / 1e9, 1),
            "route_plus_sort_us": round(r_us + s_us, 2), "fused_us": round(f_us, 2),
            "fused_plain_us": round(f_plain, 2),
            "fused_launches": "route, then moe_sort's launches", "num_tokens_post_pad": npp,
            "timing": "CUDA graph, 20 calls per replay"}


# sort-only workloads (T, topk, E_tot, block_m, Zipf skew of the expert load):
# the prefill shape, the large-E shape and about a million pairs
SORT_SCALING = ((16384, 9, 385, 64, 1.1), (8192, 36, 2304, 64, 0.8), (131072, 8, 256, 32, 1.1))


def sort_scaling(mr, dev, stream, reps=20, shapes=SORT_SCALING) -> dict:
    """moe_sort alone on seeded (token, slot) -> expert assignments of growing
    size, to show how its cost grows with T*topk. CUDA-graph replays."""
    L = mr._lib
    s = stream.cuda_stream
    out = {"timing": f"CUDA graph, {reps} calls per replay"}
    for T, k, E_tot, bm, skew in shapes:
        idx, wt = synth.random_topk_idx(T, k, E_tot, skew)
        idx, wt = idx.to(dev), wt.to(dev)
        bufs = mr.sort_buffers(T, k, E_tot, bm, dev)
        ws = torch.empty(max(1, mr.moe_sort_workspace_bytes(T, k, E_tot, bm)), dtype=torch.uint8, device=dev)
        a = [bufs[n].data_ptr() for n in ("sorted_token_ids", "sorted_weights", "expert_ids", "num_tokens_post_pad")]

        def call(idx=idx, wt=wt, a=a, ws=ws, bufs=bufs, T=T, k=k, E_tot=E_tot, bm=bm):
            rc = L.moe_sort(idx.data_ptr(), wt.data_ptr(), T, k, E_tot, bm, a[0], a[1], a[2], a[3], ws.data_ptr(),
                            ws.numel(), None, s)
            if rc != 0:
                raise RuntimeError(mr.strerror(rc))

        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
        torch.cuda.synchronize()
        us = graph_us(call, stream, reps)
        with plain_order(mr):
            us_plain = graph_us(call, stream, reps)
        out[f"T={T} k={k} E_tot={E_tot} bm={bm}"] = {"pairs": T * k, "us": round(us, 2), "plain_us": round(us_plain, 2),
                                                      "ns_per_kpair": round(us * 1e6 / (T * k), 1)}
    return out


def summary(line) -> dict:
    """The key figures of the line, short enough to survive a truncated log:
    fractions of the measured HBM peak per kernel (in the step, and isolated
    with rotated buffers), decode µs (fused/unfused x graph/eager, the launch
    floor), the prefill route + sort and the sort's growth."""
    pk = line["roofline"]["peak"]
    out = {"peak_GB/s": pk, "step_frac": {n: v["frac_of_peak"] for n, v in line["per_kernel"].items()}}
    for name, d in line.get("breakdown", {}).items():
        short = name.replace("softmax_T8192_", "").replace("sigmoid_bias_T8192_", "sig_")
        short = short.replace("_isolated", "_iso")
        out[short] = [round(d[kd]["GB/s"] / pk, 2) for kd in ("fwd", "bwd", "aux_fwd", "aux_bwd") if kd in d]
    dec = line.get("decode")
    if dec:
        fl = dec["launch_floor"]
        out["decode_floor_us[g,g_plain,e]"] = [fl["graph_us"], fl.get("graph_plain_us"), fl["eager_us"]]
        out["decode_us[fg,fg_plain,fe,ug,ug_plain,ue]"] = {
            t.split("=")[1]: [dec[t]["fused_graph_us"], dec[t].get("fused_graph_plain_us"), dec[t]["fused_eager_us"],
                              dec[t]["unfused_graph_us"], dec[t].get("unfused_graph_plain_us"),
                              dec[t]["unfused_eager_us"]]
            for t in dec if t.startswith("T=") and int(t.split("=")[1]) <= 16}
    pf = line.get("prefill_route_sort")
    if pf:
        out["prefill_us[route,sort,fused,fused_plain]"] = [pf["route_us"], pf["sort_us"], pf["fused_us"],
                                                           pf["fused_plain_us"]]
    ss = line.get("sort_scaling")
    if ss:
        out["sort_us_by_pairs"] = {v["pairs"]: v["us"] for k, v in ss.items() if isinstance(v, dict)}
    return out


def aux_loss_rates(mr, w, dev, stream, reps=50) -> dict:
    """The aux-loss scalar on the step's aux scores: per-expert counts of the aux
    routing map, the loss (column sums + final reduction) and its gradient."""
    _, t, _ = make_step(mr, w, dev, stream)
    L = mr._lib
    s = stream.cuda_stream
    T, E, k = w.T, w.E, w.topk
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    gl = torch.ones(1, dtype=torch.float32, device=dev)
    grad = torch.empty(T, E, dtype=torch.float32, device=dev)
    ws = torch.empty(mr.moe_aux_loss_workspace_bytes(T, E), dtype=torch.uint8, device=dev)
    L.moe_aux_scores_fwd(T, E, k, w.score_fn, w.in_dtype, t["x"].data_ptr(), t["scores"].data_ptr(),
                         t["amap"].data_ptr(), s)
    calls = {
        "tokens_per_expert": lambda: L.moe_tokens_per_expert(T, E, t["amap"].data_ptr(), counts.data_ptr(), s),
        "loss_fwd": lambda: L.moe_aux_loss_fwd(T, E, k, 0.01, T, t["scores"].data_ptr(), counts.data_ptr(),
                                               loss.data_ptr(), ws.data_ptr(), ws.numel(), s),
        "loss_bwd": lambda: L.moe_aux_loss_bwd(T, E, k, 0.01, T, counts.data_ptr(), gl.data_ptr(), grad.data_ptr(), s),
    }
    nbytes = {"tokens_per_expert": T * E + E * 4, "loss_fwd": T * E * 4 + E * 4 + 4, "loss_bwd": T * E * 4 + E * 4 + 4}
    # each call is ~10-30 µs, about as long as launching it from Python, so the
    # calls are captured into a CUDA graph (20 back to back) and the replays timed
    with torch.cuda.stream(stream):
        for _ in range(3):
            for fn in calls.values():
                fn()
    torch.cuda.synchronize()
    pk = peaks()["hbm_gbs"]
    out = {"workload": f"T={T} E={E} topk={k} aux scores of the step", "timing": "CUDA graph, 20 calls per replay"}
    for n, fn in calls.items():
        with plain_order(mr):
            us = graph_us(fn, stream, 20, max(1, reps // 10))
        gbs = nbytes[n] / (us * 1e-6) / 1e9
        out[n] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / pk, 3)}
    return out


def e2e_rate(mr, w, dev, stream, steps=10) -> dict:
    """The same step through the C ABI with host buffers: every step copies its
    inputs in from pinned host memory and reads every output back. Steps are
    pipelined the way a caller would run them: two device buffer sets, the
    host-to-device copies on one stream, the kernels on `stream`, the
    device-to-host copies on a third, ordered by events (a step's inputs land
    while the previous step computes and the one before is read back)."""
    sets = [make_step(mr, w, dev, stream)[:2] for _ in range(2)]
    outs = ("probs", "map", "inter", "idx", "w", "dx", "scores", "amap", "adx")
    t0 = sets[0][1]
    host_in = {n: t0[n].cpu().pin_memory() for n in ("x", "g")}
    host_out = {n: torch.empty(t0[n].shape, dtype=t0[n].dtype).pin_memory() for n in outs}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    out_done = [None, None]

    def one(i):
        launches, t = sets[i % 2]
        with torch.cuda.stream(s_in):
            if out_done[i % 2] is not None:  # this set's previous step has been read back
                s_in.wait_event(out_done[i % 2])
            for n, h in host_in.items():
                t[n].copy_(h, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        stream.wait_event(in_done)
        with torch.cuda.stream(stream):
            for _, fn in launches:
                fn()
            comp_done = torch.cuda.Event()
            comp_done.record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done)
            for n in outs:
                host_out[n].copy_(t[n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_out)
            out_done[i % 2] = ev

    one(0)
    one(1)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        one(i)
    b.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nb = sum(step_bytes(w).values())
    return {"value": round(nb / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "2 buffer sets; h2d / kernels / d2h on 3 streams; timed over %d steps" % steps}


# ---------------------------------------------------------------------------------------- CPU oracle


def _oracle_step(oracle, w, x, g):
    o = oracle.router_fwd(x, w.topk, w.score_fn, w.renorm, 0, 0, 0, w.scaling, 1.0, None)
    oracle.router_bwd(g, o["intermediate"], o["routing_map"], w.score_fn, w.renorm, w.scaling)
    a = oracle.aux_scores_fwd(x, w.topk, w.score_fn)
    oracle.aux_scores_bwd(g, a["scores"], w.score_fn)


def oracle_step_sample(w, rows: int, threads: int = 1) -> tuple[float, int, str]:
    """Times the oracle over `rows` token rows of the step's workload; returns
    (seconds, algorithmic bytes of the sample, description). With threads > 1
    the rows are split into that many contiguous slices and each thread runs
    the same oracle calls on its slice (the oracle's C functions keep no state
    between calls, and ctypes releases the GIL while they run)."""
    import oracle

    oracle.build()
    x = w.make_logits()[:rows].float().numpy()
    g = synth.grad(w.T, w.E)[:rows].double().numpy()
    if threads <= 1:
        t0 = time.perf_counter()
        _oracle_step(oracle, w, x, g)
        dt = time.perf_counter() - t0
        how = "single-threaded C oracle"
    else:
        b = np.linspace(0, rows, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as ex:
            t0 = time.perf_counter()
            list(ex.map(lambda i: _oracle_step(oracle, w, x[b[i]:b[i + 1]], g[b[i]:b[i + 1]]), range(threads)))
            dt = time.perf_counter() - t0
        how = f"C oracle on {threads} threads, one contiguous slice of rows each"
    sub = synth.Workload(w.name, rows, w.E, w.topk, w.score_fn, w.in_dtype)
    nb = sum(step_bytes(sub).values())
    return dt, nb, f"{rows} of {w.T} token rows of the step (fwd+bwd+aux fwd+aux bwd), {how}"


def cpu_baseline(w, rows: int, reps: int = 5) -> dict:
    """The oracle single-threaded (the reported baseline) and token-parallel
    over every host core, each the median of `reps` runs after one warm-up."""
    def timed(threads):
        oracle_step_sample(w, rows, threads)  # warm-up
        runs = [oracle_step_sample(w, rows, threads) for _ in range(reps)]
        return statistics.median(r[0] for r in runs), runs[0][1], runs[0][2]

    dt, nb, desc = timed(1)
    out = {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{desc}; median of {reps} runs after 1 warm-up", "seconds": round(dt, 3)}
    ncores = os.cpu_count() or 1
    if ncores > 1:
        dtp, nbp, descp = timed(ncores)
        out["parallel"] = {"value": round(nbp / dtp / 1e9, 4), "unit": "GB/s", "cores": ncores, "kind": "oracle",
                           "sample": f"{descp}; median of {reps} runs after 1 warm-up", "seconds": round(dtp, 3)}
    return out


# ---------------------------------------------------------------------------------------- main


# --workload choices for the timed step (the default is the headline workload;
# the others exist for profiling captures of the same kernels on other shapes)
STEP_WORKLOADS = {
    "softmax_T8192_E2304_k36": synth.large_e_softmax,
    "sigmoid_bias_T8192_E2304_k36": synth.large_e_sigmoid,
    **{f"softmax_T8192_E512_k{k}": (lambda k=k: synth.large_softmax(k)) for k in synth.LARGE_TOPKS},
}


def aggregate_over_ranks(elapsed_ms: float, bytes_per_step: int, steps: int, ws: int, device) -> tuple:
    """Whole-job figures of a timed region that every rank ran on its own batch:
    the elapsed time is the maximum over ranks (all_reduce MAX on the process
    group, which must be initialised when ws > 1), and the rate counts the
    bytes of all ranks. Returns (elapsed_ms, ms_per_step, GB/s)."""
    if ws > 1:
        import torch.distributed as dist

        tt = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        elapsed_ms = float(tt.item())
    value = bytes_per_step * steps * ws / (elapsed_ms * 1e-3) / 1e9
    return elapsed_ms, elapsed_ms / steps, value


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = synth.large_e_softmax()
    # rows per step sized so that warmup + steps take about args.ref_seconds
    t64, _, _ = oracle_step_sample(w, 64)
    per_step = args.ref_seconds / max(1, args.warmup + args.steps)
    rows = int(max(8, min(w.T, 64 * per_step / max(t64, 1e-6))))
    times = []
    for i in range(args.warmup + args.steps):
        dt, nb, desc = oracle_step_sample(w, rows)
        if i >= args.warmup:
            times.append(dt)
    dt = sum(times) / len(times)
    value = nb / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.workload == "softmax_T8192_E2304_k36" else args.workload,
                       "T": w.T, "E": w.E, "topk": w.topk,
                       "score_fn": "softmax" if w.score_fn == synth.SOFTMAX else "sigmoid",
                       "sample_rows_per_step": rows},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["all", "step", "decode", "aux_loss", "prefill", "bf16", "sort"], default="all",
                    help="step: the timed step only; decode: the decode latency table only "
                         "(both used for profiling captures)")
    ap.add_argument("--decode-calls", type=int, default=200, help="calls per decode timing loop")
    ap.add_argument("--decode-ts", default=",".join(str(t) for t in synth.DECODE_BENCH_TS),
                    help="decode token counts, comma separated")
    ap.add_argument("--workload", choices=sorted(STEP_WORKLOADS), default="softmax_T8192_E2304_k36",
                    help="workload of the timed step (default: the headline one)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=8192, help="oracle sample size (token rows)")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="reference arm: CPU time budget for warmup + steps")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    ws, rank, local = dist_env()
    import top_gating_expert_row_gb300 as mr

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the routing path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.only == "decode":
        if rank == 0:
            ts = tuple(int(t) for t in args.decode_ts.split(","))
            print(json.dumps({"decode_gpt_oss": decode_latency(mr, dev, torch.cuda.Stream(device=dev),
                                                               args.decode_calls, (1, 4, 16, 32, 64, 128, 256),
                                                               synth.decode_gpt_oss)}), flush=True)
            print(json.dumps({"decode": decode_latency(mr, dev, torch.cuda.Stream(device=dev),
                                                       args.decode_calls, ts)}), flush=True)
        return 0
    if args.only == "bf16":
        if rank == 0:
            print(json.dumps({"bf16": bf16_rates(mr, dev, torch.cuda.Stream(device=dev))}), flush=True)
        return 0
    if args.only == "sort":
        if rank == 0:
            print(json.dumps({"sort_scaling": sort_scaling(mr, dev, torch.cuda.Stream(device=dev))}), flush=True)
        return 0
    if args.only == "prefill":
        if rank == 0:
            print(json.dumps({"prefill_route_sort": prefill_route_sort(mr, dev, torch.cuda.Stream(device=dev))}),
                  flush=True)
        return 0
    if args.only == "aux_loss":
        if rank == 0:
            print(json.dumps({"aux_loss": aux_loss_rates(mr, dev=dev, w=STEP_WORKLOADS[args.workload](),
                                                         stream=torch.cuda.Stream(device=dev))}), flush=True)
        return 0
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(device=dev)
    w = STEP_WORKLOADS[args.workload]()
    launches, _t, _ = make_step(mr, w, dev, stream)
    nbytes = step_bytes(w)
    tm = Timer(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for _, fn in launches:
                fn()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            for name, fn in launches:
                tm.around(name, fn)
        end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    elapsed_ms, ms_per_step, value = aggregate_over_ranks(start.elapsed_time(end), sum(nbytes.values()), args.steps,
                                                          ws, dev)

    pk = peaks()
    per_kernel = {}
    for name, nb in nbytes.items():
        ms = tm.mean_ms(name)
        per_kernel[name] = {"us": round(ms * 1e3, 2), "GB/s": round(nb / (ms * 1e-3) / 1e9, 1),
                            "frac_of_peak": round(nb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3),
                            "page_B300_GB/s": PAGE_B300.get(
                                (name, "softmax" if w.score_fn == synth.SOFTMAX else "sigmoid", w.E, w.topk))}
    dom = max(per_kernel, key=lambda n: per_kernel[n]["us"])
    dom_ms = tm.mean_ms(dom)
    achieved = nbytes[dom] / (dom_ms * 1e-3) / 1e9
    traffic = profiled_traffic() if dom == "fwd" else None
    fwd_kernel = "k_router_fwd_wide" if w.E > 1024 else "k_router_fwd"
    roofline = {"kernel": {"fwd": fwd_kernel, "bwd": "k_router_bwd", "aux_fwd": f"{fwd_kernel} (aux scores)",
                           "aux_bwd": "k_router_bwd (aux scores)"}[dom],
                "bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 3), "peak_source": pk["source"] + " (hbm_gbs)",
                "traffic": traffic, "algorithmic_bytes": nbytes[dom]}

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD if args.workload == "softmax_T8192_E2304_k36" else args.workload,
                       "T": w.T, "E": w.E, "topk": w.topk,
                       "score_fn": "softmax" if w.score_fn == synth.SOFTMAX else "sigmoid",
                       "kernels_per_step": [n for n, _ in launches], "bytes_per_step": sum(nbytes.values()),
                       "l2": "no flush; inputs larger than L2 (each step touches ~565 MB against 129 MB of L2)",
                       "parallelism": f"replicas x{ws} (tokens are independent; no collective)"},
            "roofline": roofline, "per_kernel": per_kernel,
            "gpu_launches": len(launches) * args.steps, "clocks": clocks}
    if args.only == "all":
        line["e2e"] = e2e_rate(mr, w, dev, stream)
        if rank == 0:
            line["decode"] = decode_latency(mr, dev, stream, args.decode_calls)
            line["decode_gpt_oss"] = decode_latency(mr, dev, stream, args.decode_calls, (1, 4, 16, 32, 64, 128, 256),
                                                    synth.decode_gpt_oss)
            line["prefill_route_sort"] = prefill_route_sort(mr, dev, stream)
            line["sort_scaling"] = sort_scaling(mr, dev, stream)
            line["aux_loss"] = aux_loss_rates(mr, w, dev, stream)
            line["bf16"] = bf16_rates(mr, dev, stream)
            breakdown = {}
            for wl in [synth.large_softmax(k) for k in synth.LARGE_TOPKS] + [synth.large_e_sigmoid(),
                                                                             synth.widest_softmax()]:
                breakdown[wl.name] = time_kernels(mr, wl, dev, stream)
            # the step's own kernels isolated: rotated buffer sets beyond L2, so the
            # backward kernels read inputs the forward did not just leave in L2
            breakdown[w.name + "_isolated"] = time_kernels(mr, w, dev, stream)
            line["breakdown"] = breakdown
            if not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(w, args.cpu_rows)
            line["summary"] = summary(line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
