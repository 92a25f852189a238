#!/usr/bin/env python3
"""Benchmark of the routed MoE prefill layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

One step is one whole layer call (moe_layer_forward: plan -> gather ->
gate/up -> down -> combine) over one synthetic chunk already resident in HBM,
on the full page-1-scale layer: T=2048 tokens, d=2560, E=512 experts, top-10,
expert FFN f=512, tm=16, skewed routing (router logits N(0,1) plus a
per-expert N(0,1) bias).  L2 is flushed (256 MiB write) before every timed
step; the weights alone (4 GB) are far larger than L2 too.

Printed: ONE JSON line with rows/s (T*k routed rows per layer), the plan's
microseconds per layer, per-stage times, the roofline of the dominant kernel
(the gate/up GEMM), the end-to-end rows/s through host buffers, SM clocks
sampled during the timed region, and the CPU oracle timed on a bounded
sample on this host's cores, and how far the layer lands from the oracle
(accuracy_vs_oracle).  Beside them: the plan alone on 1M and 10M entries
(plan_sweep), the plan + gather configuration with fp16 rows (plan_gather),
the same layer on 8-bit operands (fp8_layer) and on MXFP4 4-bit weights
(mxfp4_layer), each with its own error against the fp64 oracle, and every
other layer workload timed the same way (workloads:
the tiny layer, the 256-expert layer, and the long prompt as its 8 chunks of
4096 tokens per step), each with per-stage times, its gate/up roofline and
the oracle on this host's cores.

``--impl reference`` times the CPU oracle itself (the only reference this
method has) on bounded samples of the same workload.

Multi-GPU (torchrun, or ``--gpus N`` alone, which starts the N ranks through
torchrun on this node): every rank runs its own independent layer on its own
chunk of tokens (weak scaling, no collective on the data path); rank 0
prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import datetime as dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_prefill_routing_gb300 import binding as B  # noqa: E402
from moe_prefill_routing_gb300 import replicas  # noqa: E402
from moe_prefill_routing_gb300 import workload as W  # noqa: E402

METRIC = "MoE layer routed rows/s (plan+gather+FFN+combine); plan µs/layer at T=2048"
WORKLOAD = 3  # the full page-1-scale layer
ROUTING = {"topk": "top-k of N(0,1) logits", "topk_bias": "top-k of N(0,1) logits + N(0,1) expert bias",
           "zipf": "Zipf (rank^-1.2) popularity, k distinct experts per token"}
# plan (one cluster launch at this size), gather, gate/up, down, combine
KERNELS_PER_LAYER = 5
FLUSH_BYTES = 256 << 20
PROFILE = os.path.join(ROOT, "profiles", "ffn_gate_up_layer_t2048_d2560_e512_k10_f512.md")
PROFILE_F8 = os.path.join(ROOT, "profiles", "ffn_gate_up_f8_layer_t2048_d2560_e512_k10_f512.md")
FFN_SRC = os.path.join(ROOT, "moe_prefill_routing_gb300", "csrc", "ffn.cu")
FALLBACK_HBM_GBS = 6800.0


# ---- helpers ----------------------------------------------------------------

def log(*a):
    print(*a, file=sys.stderr, flush=True)


FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    """(HBM GB/s, bf16 TFLOP/s for a kernel timed alone, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def profile_traffic(path=PROFILE):
    """dram bytes per launch of the gate/up kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    h = re.search(r"ffn_cu_sha256:\s*([0-9a-f]{64})", txt)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(FFN_SRC, "rb").read()).hexdigest()
    return int(m.group(1)) if h.group(1) == cur else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            cmd.insert(1, f"--id={uuid if uuid.startswith('GPU-') else 'GPU-' + uuid}")
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            return None
        inwin = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        use = inwin or rows
        reasons = sorted({n for r in use for n, v in zip(self.NAMES, r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inwin else "whole run"}


def algorithmic(wl, ids, wbytes=2, abytes=2):
    """Algorithmic work of one layer from the routing itself: active experts,
    real and padded rows, and the bytes / flops each stage must move.
    ``wbytes`` is the size of one weight element (2 bf16, 1 E4M3, which also
    reads one fp32 scale per expert and output feature); ``abytes`` the size
    of one element of the GEMMs' row operands (2 bf16, 1 E4M3 rows of x and
    H, which also carry one int32 exponent per row)."""
    flat = ids.ravel()
    counts = np.bincount(flat[flat >= 0], minlength=wl.E)
    active = int((counts > 0).sum())
    R = int(counts.sum())
    R_pad = int((-(-counts // wl.tm) * wl.tm).sum())
    d, f = wl.d, wl.f
    sc = 4 if wbytes == 1 else 0  # E4M3 scales
    ex = 4 if abytes == 1 else 0  # E4M3 row exponents
    gate_up = (active * 2 * (d * f * wbytes + f * sc) + R_pad * (d * abytes + ex) +
               R_pad * f * 2)
    gate_up_flops = 4 * d * f * R
    down = (active * (f * d * wbytes + d * sc) + R_pad * (f * abytes + ex) + R_pad * d * 2 +
            R_pad * 4)
    if abytes == 1:  # the pass that turns H into E4M3 rows
        down += R_pad * f * 2 + R_pad * (f + ex)
    gather = wl.T * d * 2 + R_pad * (d * abytes + ex) + R_pad * 4
    combine = R * d * 2 + wl.T * d * 2 + R * 4
    plan = 8 * wl.T * wl.k + 4 * wl.T * wl.k + 8 * R_pad + 8 * (wl.E + 1)
    return dict(active=active, R=R, R_pad=R_pad, gate_up=gate_up, gate_up_flops=gate_up_flops,
                down=down, gather=gather,
                combine=combine, plan=plan, layer=plan + gather + gate_up + down + combine,
                flops=6 * d * f * R, weights=active * 3 * d * f * wbytes)


def d16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


# ---- CPU oracle timing ----------------------------------------------------------

def oracle_sample(inp, wl, budget_s, nthreads, with_output=False):
    """Times the oracle on a bounded sample of the workload: the full plan
    (single-threaded by definition) and the layer for the first n tokens,
    n chosen to take about budget_s.  Returns rows/s and a description."""
    import oracle  # CPU baseline leg only

    t = time.perf_counter()
    oracle.plan(inp["ids"], inp["w"], wl.E, wl.tm)
    t_plan = time.perf_counter() - t
    args = (inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    pilot = np.arange(min(4, wl.T), dtype=np.int32)
    t = time.perf_counter()
    oracle.layer(*args, x_dtype=wl.x_dtype, tokens=pilot, nthreads=nthreads)
    per_tok = (time.perf_counter() - t) / len(pilot)
    n = int(max(len(pilot), min(wl.T, budget_s / max(per_tok, 1e-9))))
    toks = np.arange(n, dtype=np.int32)
    t = time.perf_counter()
    y_ref = oracle.layer(*args, x_dtype=wl.x_dtype, tokens=toks, nthreads=nthreads)
    t_layer = time.perf_counter() - t
    secs = t_layer + t_plan * n / wl.T
    rows = n * wl.k
    if with_output:
        return rows / secs, secs, _sample_desc(wl, n, rows, nthreads), toks, y_ref
    return rows / secs, secs, _sample_desc(wl, n, rows, nthreads)


def _sample_desc(wl, n, rows, nthreads):
    return (f"plan of all {wl.T * wl.k} rows (1 thread) + fp64 FFN/combine of the first {n} "
            f"tokens ({rows} rows) on {nthreads} threads; plan time prorated per row")


def error_vs_oracle(y_dev, toks, y_ref):
    """max |y - oracle| and rel-L2 on the oracle's tokens, with the layer bound
    1e-2 * max|oracle| + 1e-3."""
    y = y_dev.float().cpu().numpy().astype(np.float64)[toks]
    err = float(np.max(np.abs(y - y_ref)))
    nrm = float(np.linalg.norm(y_ref))
    return {"tokens": int(len(toks)), "max_abs_err": err,
            "rel_l2": float(np.linalg.norm(y - y_ref)) / nrm if nrm > 0 else 0.0,
            "bound": 1e-2 * float(np.max(np.abs(y_ref))) + 1e-3}


# ---- native arm ------------------------------------------------------------------

def run_native(args, rank, world, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.workload(args.workload)
    chunk = replicas.chunk_of_rank(rank, world) % wl.n_chunks
    log(f"[rank {rank}] generating {wl.name} (chunk {chunk}) ...")
    inp = W.make_inputs(wl, seed=0, chunk=chunk)
    f8 = args.weights == "f8"
    e4m3 = args.weights == "e4m3" or f8
    alg = algorithmic(wl, inp["ids"], wbytes=1 if e4m3 else 2, abytes=1 if f8 else 2)
    x, ids, w = d16(inp["x"], dev), torch.from_numpy(inp["ids"]).to(dev), torch.from_numpy(inp["w"]).to(dev)
    Wg, Wu, Wd = (d16(inp[n], dev) for n in ("Wg", "Wu", "Wd"))
    if e4m3:
        # the experts' weights as E4M3 codes + per-feature scales (quantized
        # once on the device, before anything is timed)
        layer = B.MoeLayer.quantized(Wg, Wu, Wd, tm=wl.tm, act_e4m3=f8)
        Wg, Wu, Wd = layer.Wg, layer.Wu, layer.Wd
        torch.cuda.synchronize(dev)
    else:
        layer = B.MoeLayer(Wg, Wu, Wd, tm=wl.tm)
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    rows = wl.T * wl.k

    def timed(step_fn, K):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            step_fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]

    # warm-up, then EXACTLY K timed layer steps
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        layer.forward(x, ids, w, y=y)
    torch.cuda.synchronize(dev)
    status = B.read_status(layer._ws)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after warm-up")
    clocks = ClockSampler(dev) if rank == 0 else None
    replicas.barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ms = timed(lambda: layer.forward(x, ids, w, y=y), args.steps)
    torch.cuda.synchronize(dev)
    replicas.barrier(world)
    t1 = time.time()
    clk = clocks.stop(t0, t1) if clocks else None
    total_ms = replicas.max_over_ranks(sum(ms), world, dev)
    value = args.steps * rows * world / (total_ms / 1e3)

    # per-stage breakdown through the stage entry points (same stream)
    cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
    o = B.plan(ids, w, wl.E, wl.tm, cap=cap)
    xs = B.gather(x, o["srt_tok"], o["offsets"], wl.E, cap)
    H = torch.empty((cap, wl.f), dtype=torch.bfloat16, device=dev)
    Ys = torch.empty((cap, wl.d), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stages = ("plan", "gather", "gate_up", "down", "combine")
    if f8:
        x8, xe = B.gather_e4m3(x, o["srt_tok"], o["offsets"], wl.E, cap)
        H8, he = B.rows_e4m3(H, o["offsets"], wl.E, cap)

        def down_f8():
            B.rows_e4m3(H, o["offsets"], wl.E, cap, H8, he)
            B.ffn_down_f8(H8, he, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys, status=st)

        calls = (lambda: B.plan(ids, w, wl.E, wl.tm, cap=cap, out=o),
                 lambda: B.gather_e4m3(x, o["srt_tok"], o["offsets"], wl.E, cap, x8, xe),
                 lambda: B.ffn_gate_up_f8(x8, xe, Wg, Wu, o["offsets"], cap, H=H, status=st),
                 down_f8,
                 lambda: B.combine(Ys, o["pos"], y=y))
    else:
        calls = (lambda: B.plan(ids, w, wl.E, wl.tm, cap=cap, out=o),
                 lambda: B.gather(x, o["srt_tok"], o["offsets"], wl.E, cap, xs=xs),
                 (lambda: B.ffn_gate_up_e4m3(xs, Wg, Wu, o["offsets"], cap, H=H, status=st)) if e4m3
                 else (lambda: B.ffn_gate_up(xs, Wg, Wu, o["offsets"], cap, H=H, status=st)),
                 (lambda: B.ffn_down_e4m3(H, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys, status=st))
                 if e4m3 else (lambda: B.ffn_down(H, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys,
                                                   status=st)),
                 lambda: B.combine(Ys, o["pos"], y=y))
    K2 = max(3, min(args.steps, 200))
    per = {s: [] for s in stages}
    for i in range(K2 + 3):
        flush.fill_(i & 0xFF)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
        ev[0].record(stream)
        for j, c in enumerate(calls):
            c()
            ev[j + 1].record(stream)
        torch.cuda.synchronize(dev)
        if i >= 3:
            for j, s in enumerate(stages):
                per[s].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
    # the plan alone, 48 layers per CUDA graph replay (the pages' plan figure is
    # a 48-layer graph median per layer); inputs stay in L2 between layers
    plan_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(plan_graph):
        for _ in range(48):
            B.plan(ids, w, wl.E, wl.tm, cap=cap, out=o)
    plan_graph.replay()
    torch.cuda.synchronize(dev)
    reps = 50
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        plan_graph.replay()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    plan_graph_us = g0.elapsed_time(g1) * 1e3 / (48 * reps)
    stage_us = {s: statistics.median(v) for s, v in per.items()}
    stage_mean_us = {s: statistics.mean(v) for s, v in per.items()}

    # end to end through the C ABI's host entry point (moe_prefill_forward_host):
    # every step copies its chunk's x, ids and w in from pinned host memory and
    # its y back out; one call runs K3 steps, so step s+1's copies in and step
    # s-1's copy out overlap step s's layer on the copy engines
    x_h = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_h = torch.from_numpy(inp["ids"]).pin_memory()
    w_h = torch.from_numpy(inp["w"]).pin_memory()
    y_h = torch.empty((wl.T, wl.d), dtype=torch.bfloat16).pin_memory()
    layer.forward_host_chunks([x_h] * 3, [ids_h] * 3, [w_h] * 3, [y_h] * 3)
    torch.cuda.synchronize(dev)
    K3 = max(3, min(args.steps, 200))
    replicas.barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.forward_host_chunks([x_h] * K3, [ids_h] * K3, [w_h] * K3, [y_h] * K3)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if B.read_status(layer._host_ws) != 0:
        raise RuntimeError("device status set in the end-to-end run")
    e2e_ms = e0.elapsed_time(e1)
    e2e_total = replicas.max_over_ranks(e2e_ms, world, dev)
    e2e_value = K3 * rows * world / (e2e_total / 1e3)
    # the same steps one call each: nothing overlaps, the copies show in full
    ms_serial = timed(lambda: layer.forward_host(x_h, ids_h, w_h, y_h), K3)
    serial_total = replicas.max_over_ranks(sum(ms_serial), world, dev)
    e2e_serial_value = K3 * rows * world / (serial_total / 1e3)
    h2d = x_h.numel() * 2 + ids_h.numel() * 4 + w_h.numel() * 4
    d2h = y_h.numel() * 2

    # alongside the bf16 measurement: the same layer with E4M3 weights and E4M3
    # activations (both GEMMs on tcgen05 kind::f8f6f4), timed the same way;
    # a different arithmetic, so reported beside the headline, not as it
    fp8 = None
    if not e4m3 and not args.no_fp8:
        layer8 = B.MoeLayer.quantized(Wg, Wu, Wd, tm=wl.tm, act_e4m3=True)
        for i in range(args.warmup):
            flush.fill_(i & 0xFF)
            layer8.forward(x, ids, w, y=y)
        torch.cuda.synchronize(dev)
        if B.read_status(layer8._ws) != 0:
            raise RuntimeError("device status set in the E4M3 layer")
        ms8 = timed(lambda: layer8.forward(x, ids, w, y=y), args.steps)
        total8 = replicas.max_over_ranks(sum(ms8), world, dev)
        y8 = layer8.forward(x, ids, w).clone()
        alg8 = algorithmic(wl, inp["ids"], wbytes=1, abytes=1)
        fp8 = {"value": args.steps * rows * world / (total8 / 1e3), "unit": "rows/s",
               "ms_per_step": statistics.mean(ms8), "steps": args.steps,
               "arithmetic": "E4M3 weights (fp32 scale per expert and output feature) and "
                             "E4M3 rows of x and H (power-of-two scale per row); fp32 "
                             "accumulation; bf16 H, Ys, y",
               "layer_hbm_gbs": alg8["layer"] / (statistics.mean(ms8) / 1e3) / 1e9,
               "gpu_launches": (KERNELS_PER_LAYER + 1) * args.steps}
        del layer8

    # MXFP4 expert weights (4-bit E2M1 codes, power-of-two scale per 32 along
    # K; decoded to bf16 into tensor memory, bf16 activations), timed the same way
    mx4 = None
    if not e4m3 and not args.no_fp8:
        layer4 = B.MoeLayer.quantized_mxfp4(Wg, Wu, Wd, tm=wl.tm)
        for i in range(args.warmup):
            flush.fill_(i & 0xFF)
            layer4.forward(x, ids, w, y=y)
        torch.cuda.synchronize(dev)
        if B.read_status(layer4._ws) != 0:
            raise RuntimeError("device status set in the MXFP4 layer")
        ms4 = timed(lambda: layer4.forward(x, ids, w, y=y), args.steps)
        total4 = replicas.max_over_ranks(sum(ms4), world, dev)
        y4 = layer4.forward(x, ids, w).clone()
        o4 = B.plan(ids, w, wl.E, wl.tm, cap=cap)
        xs4 = B.gather(x, o4["srt_tok"], o4["offsets"], wl.E, cap)
        H4 = torch.empty((cap, wl.f), dtype=torch.bfloat16, device=dev)
        Ys4 = torch.empty((cap, wl.d), dtype=torch.bfloat16, device=dev)
        gu4, dn4 = [], []
        for i in range(min(args.steps, 50) + 3):
            flush.fill_(i & 0xFF)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            B.ffn_gate_up_mxfp4(xs4, layer4.Wg, layer4.Wu, o4["offsets"], cap, H=H4)
            ev[1].record(stream)
            B.ffn_down_mxfp4(H4, layer4.Wd, o4["offsets"], o4["srt_w"], cap, Ys=Ys4)
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                gu4.append(ev[0].elapsed_time(ev[1]) * 1e3)
                dn4.append(ev[1].elapsed_time(ev[2]) * 1e3)
        mx4 = {"value": args.steps * rows * world / (total4 / 1e3), "unit": "rows/s",
               "ms_per_step": statistics.mean(ms4), "steps": args.steps,
               "gate_up_us": statistics.median(gu4), "down_us": statistics.median(dn4),
               "arithmetic": "MXFP4 weights (4-bit E2M1 codes, power-of-two scale per 32 along "
                             "K, decoded exactly to bf16 into tensor memory); bf16 activations, "
                             "fp32 accumulation; bf16 H, Ys, y",
               "weight_bytes_active": alg["active"] * 3 * wl.d * wl.f // 2,
               "gpu_launches": KERNELS_PER_LAYER * args.steps}
        del layer4, o4, xs4, H4, Ys4

    # the plan alone on large inputs, where its HBM traffic is what bounds it:
    # T*k = 1M and 10M entries, E = 512, ids uniform over the experts (drawn on
    # the device from a seeded generator), L2 flushed before each call
    sweep = None
    if not args.no_plan_sweep:
        sweep = []
        hbm_peak = peaks()[0]
        for n in (1 << 20, 10 << 20):
            kk, EE, tmm = 10, 512, 16
            TT = n // kk
            gen = torch.Generator(device=dev).manual_seed(1234 + n)
            ids_s = torch.randint(0, EE, (TT, kk), generator=gen, device=dev, dtype=torch.int32)
            w_s = torch.rand((TT, kk), generator=gen, device=dev)
            cap_s = B.capacity(TT, kk, EE, tmm)
            o_s = B.plan(ids_s, w_s, EE, tmm, cap=cap_s)
            ts = []
            for i in range(13):
                flush.fill_(i & 0xFF)
                a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_ev.record(stream)
                B.plan(ids_s, w_s, EE, tmm, cap=cap_s, out=o_s)
                b_ev.record(stream)
                torch.cuda.synchronize(dev)
                if i >= 3:
                    ts.append(a_ev.elapsed_time(b_ev) * 1e3)
            r_pad = int(o_s["offsets"][-1])
            # read ids and w, write pos, srt_tok and srt_w, the offsets and counts
            byts = 8 * n + 4 * n + 8 * r_pad + 8 * (EE + 1)
            us = statistics.median(ts)
            sweep.append({"entries": n, "T": TT, "k": kk, "E": EE, "tm": tmm, "us": us,
                          "algorithmic_bytes": byts, "hbm_gbs": byts / us / 1e3,
                          "frac": byts / us / 1e3 / hbm_peak})
            del ids_s, w_s, o_s

    # the plan + gather configuration (no expert FFN): T=2048, E=512, top-10,
    # d=2560 fp16 rows gathered into expert order; each step = one moe_plan
    # and one moe_gather on inputs resident in HBM, L2 flushed before it
    plan_gather = None
    if not args.no_plan_gather:
        wl2 = W.workload(2)
        inp2 = W.make_inputs(wl2, seed=0, weights=False)
        x2 = torch.from_numpy(np.ascontiguousarray(inp2["x"]).view(np.int16)).to(dev).view(
            torch.float16)
        ids2 = torch.from_numpy(inp2["ids"]).to(dev)
        w2 = torch.from_numpy(inp2["w"]).to(dev)
        cap2 = B.capacity(wl2.T, wl2.k, wl2.E, wl2.tm)
        o2 = B.plan(ids2, w2, wl2.E, wl2.tm, cap=cap2)
        xs2 = B.gather(x2, o2["srt_tok"], o2["offsets"], wl2.E, cap2)

        def plan_step():
            B.plan(ids2, w2, wl2.E, wl2.tm, cap=cap2, out=o2)

        def gather_step():
            B.gather(x2, o2["srt_tok"], o2["offsets"], wl2.E, cap2, xs=xs2)

        def both():
            plan_step()
            gather_step()

        for i in range(args.warmup):
            flush.fill_(i & 0xFF)
            both()
        torch.cuda.synchronize(dev)
        K2 = min(args.steps, 200)
        ms2 = timed(both, K2)
        g_ms = timed(gather_step, K2)
        r_pad2 = int(o2["offsets"][-1])
        g_us = statistics.mean(g_ms) * 1e3
        # bytes the gather must move across HBM at least once: x read once (its
        # rows are read k times, from L2 after the first), xs written, srt_tok
        g_bytes = wl2.T * wl2.d * 2 + r_pad2 * wl2.d * 2 + 4 * r_pad2
        plan_gather = {"workload": wl2.name, "x_dtype": "f16",
                       "value": wl2.T * wl2.k / (statistics.mean(ms2) / 1e3), "unit": "rows/s",
                       "ms_per_step": statistics.mean(ms2), "steps": K2, "R_pad": r_pad2,
                       "gather_us": g_us, "gather_hbm_bytes": g_bytes,
                       "gather_hbm_gbs": g_bytes / g_us / 1e3,
                       "gather_frac": g_bytes / g_us / 1e3 / peaks()[0]}
        del x2, ids2, w2, o2, xs2

    if rank != 0:
        return
    hbm, tflops, peak_src = peaks()
    if f8:  # dense fp8 tensor peak: the measured bf16 figure x the nominal 2x ratio
        tflops *= 2.0
        peak_src += " (fp8 = 2 x bf16)"
    t_gu = stage_mean_us["gate_up"] * 1e-6
    # the bound is whichever of the two floors is longer for this kernel
    tensor_bound = alg["gate_up_flops"] / (tflops * 1e12) > alg["gate_up"] / (hbm * 1e9)
    if tensor_bound:
        achieved, peak, unit = alg["gate_up_flops"] / t_gu / 1e12, tflops, "TFLOP/s"
    else:
        achieved, peak, unit = alg["gate_up"] / t_gu / 1e9, hbm, "GB/s"
    traffic = profile_traffic(PROFILE_F8 if f8 else PROFILE)
    layer_gbs = alg["layer"] / (sum(ms) / len(ms) / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 x e4m3 -> f32 (weights and activations)" if f8 else
                  "bf16 (E4M3 weights widened to bf16)" if e4m3 else "bf16"),
        "data": "synthetic (seeded: x~N(0,1), W~N(0,0.02) bf16, " + ROUTING[wl.routing] + ")",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "f": wl.f,
                   "tm": wl.tm, "routing": ROUTING[wl.routing],
                   "active_experts": alg["active"], "R_pad": alg["R_pad"],
                   "weights": ("E4M3 codes + fp32 scale per expert and output feature" if e4m3
                               else "bf16"),
                   "activations": ("E4M3 rows of x and H, power-of-two scale per row" if f8
                                   else "bf16"),
                   "l2": "flushed before every timed step (256 MiB write)",
                   "parallelism": "replicas (one independent layer per GPU)"},
        "plan_us_per_layer": plan_graph_us,
        "plan_us_per_layer_method": "48 moe_plan calls per CUDA graph replay, mean per call",
        "plan_us_cold": stage_us["plan"],
        "plan_sweep": sweep,
        "plan_gather": plan_gather,
        "stages_us": stage_us,
        "layer_hbm_gbs": layer_gbs,
        "roofline": {"kernel": ("k_ffn<gate/up, E4M3 operands> (tcgen05.mma.kind::f8f6f4 "
                               "grouped GEMM + SwiGLU)") if f8
                     else ("k_ffn<gate/up, E4M3 weights> (widened to bf16 in shared memory; "
                           "tcgen05 grouped GEMM + SwiGLU)") if e4m3
                     else "k_ffn<gate/up> (tcgen05 grouped GEMM + SwiGLU)",
                     "bound": "tensor" if tensor_bound else "hbm",
                     "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": alg["gate_up"],
                     "algorithmic_flops_per_launch": alg["gate_up_flops"],
                     "traffic": (traffic if args.workload == WORKLOAD and (f8 or not e4m3)
                                 else None)},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_total / K3, "steps": K3,
                "api": "moe_prefill_forward_host (host buffers; copies overlap the layer)",
                "serial_value": e2e_serial_value,
                "serial_note": "one call per step, L2 flushed before each: copies not overlapped",
                "l2": "not flushed: every step streams the active expert weights "
                      f"({alg['weights'] / 1e9:.2f} GB > 129 MB L2)"},
        "clocks": clk,
        "fp8_layer": fp8,
        "mxfp4_layer": mx4,
        "gpu_launches": (KERNELS_PER_LAYER + int(f8)) * args.steps,
    }
    if world == 1 and not args.no_cpu_baseline and not e4m3:
        nth = os.cpu_count() or 1
        log("timing the CPU oracle on a bounded sample ...")
        v, secs, desc, toks, y_ref = oracle_sample(inp, wl, args.cpu_budget, nth, with_output=True)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": nth, "kind": "oracle",
                                "sample": desc, "seconds": secs}
        # how far each arithmetic lands from the fp64 oracle (bf16 weights) on
        # the oracle's tokens: the bf16 layer and, beside it, the 8-bit one
        y16 = layer.forward(x, ids, w)
        line["accuracy_vs_oracle"] = {"bf16_layer": error_vs_oracle(y16, toks, y_ref)}
        if fp8 is not None:
            fp8["accuracy_vs_oracle"] = error_vs_oracle(y8, toks, y_ref)
            line["accuracy_vs_oracle"]["fp8_layer"] = fp8["accuracy_vs_oracle"]
        if mx4 is not None:
            mx4["accuracy_vs_oracle"] = error_vs_oracle(y4, toks, y_ref)
            line["accuracy_vs_oracle"]["mxfp4_layer"] = mx4["accuracy_vs_oracle"]
    if world == 1 and not args.no_workloads and not e4m3:
        line["workloads"] = other_workloads(args, dev, flush, stream)
    print(json.dumps(line), flush=True)


# ---- the other layer workloads ------------------------------------------------------

def other_workloads(args, dev, flush, stream):
    """Every other layer workload, each timed like the headline: the tiny
    layer, the 256-expert layer and the long prompt (its 8 chunks of 4096
    tokens per step).  Per workload: routed rows/s, per-stage times, the
    gate/up kernel's roofline and the oracle on this host's cores."""
    out = {}
    hbm, tflops, peak_src = peaks()
    for idx in (1, 4, 5):
        wl = W.workload(idx)
        log(f"workload {wl.name} ...")
        chunks = [W.make_inputs(wl, seed=0, chunk=c, weights=(c == 0)) for c in range(wl.n_chunks)]
        inp = chunks[0]
        Wg, Wu, Wd = (d16(inp[n], dev) for n in ("Wg", "Wu", "Wd"))
        layer = B.MoeLayer(Wg, Wu, Wd, tm=wl.tm)
        xs_d = [d16(c["x"], dev) for c in chunks]
        ids_d = [torch.from_numpy(c["ids"]).to(dev) for c in chunks]
        w_d = [torch.from_numpy(c["w"]).to(dev) for c in chunks]
        y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device=dev)

        def step():
            for c in range(wl.n_chunks):
                layer.forward(xs_d[c], ids_d[c], w_d[c], y=y)

        for i in range(args.warmup):
            flush.fill_(i & 0xFF)
            step()
        torch.cuda.synchronize(dev)
        if B.read_status(layer._ws) != 0:
            raise RuntimeError(f"device status set in workload {wl.name}")
        K = max(3, args.steps)
        ms = []
        for i in range(K):
            flush.fill_(i & 0xFF)
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            step()
            b_ev.record(stream)
            ms.append((a_ev, b_ev))
        torch.cuda.synchronize(dev)
        ms = [a_ev.elapsed_time(b_ev) for a_ev, b_ev in ms]
        rows = wl.T * wl.k * wl.n_chunks
        # stages of chunk 0, each through its own entry point, L2 flushed first
        cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
        x0, i0, w0 = xs_d[0], ids_d[0], w_d[0]
        o = B.plan(i0, w0, wl.E, wl.tm, cap=cap)
        xs = B.gather(x0, o["srt_tok"], o["offsets"], wl.E, cap)
        H = torch.empty((cap, wl.f), dtype=torch.bfloat16, device=dev)
        Ys = torch.empty((cap, wl.d), dtype=torch.bfloat16, device=dev)
        stages = ("plan", "gather", "gate_up", "down", "combine")
        calls = (lambda: B.plan(i0, w0, wl.E, wl.tm, cap=cap, out=o),
                 lambda: B.gather(x0, o["srt_tok"], o["offsets"], wl.E, cap, xs=xs),
                 lambda: B.ffn_gate_up(xs, Wg, Wu, o["offsets"], cap, H=H),
                 lambda: B.ffn_down(H, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys),
                 lambda: B.combine(Ys, o["pos"], y=y))
        per = {st: [] for st in stages}
        for i in range(min(K, 50) + 3):
            flush.fill_(i & 0xFF)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
            ev[0].record(stream)
            for j, c in enumerate(calls):
                c()
                ev[j + 1].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                for j, st in enumerate(stages):
                    per[st].append(ev[j].elapsed_time(ev[j + 1]) * 1e3)
        stage_us = {st: statistics.median(v) for st, v in per.items()}
        alg = algorithmic(wl, inp["ids"])
        t_gu = statistics.mean(per["gate_up"]) * 1e-6
        tensor_bound = alg["gate_up_flops"] / (tflops * 1e12) > alg["gate_up"] / (hbm * 1e9)
        if tensor_bound:
            achieved, peak, unit = alg["gate_up_flops"] / t_gu / 1e12, tflops, "TFLOP/s"
        else:
            achieved, peak, unit = alg["gate_up"] / t_gu / 1e9, hbm, "GB/s"
        entry = {
            "workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "f": wl.f,
            "tm": wl.tm, "routing": ROUTING[wl.routing], "chunks_per_step": wl.n_chunks,
            "value": K * rows / (sum(ms) / 1e3), "unit": "rows/s",
            "ms_per_step": statistics.mean(ms), "steps": K,
            "active_experts_chunk0": alg["active"], "R_pad_chunk0": alg["R_pad"],
            "stages_us_chunk0": stage_us,
            "layer_hbm_gbs_chunk0": alg["layer"] / (statistics.mean(ms) / wl.n_chunks / 1e3) / 1e9,
            "roofline": {"kernel": "k_ffn<gate/up> (tcgen05 grouped GEMM + SwiGLU), chunk 0",
                         "bound": "tensor" if tensor_bound else "hbm", "achieved": achieved,
                         "peak": peak, "unit": unit, "frac": achieved / peak,
                         "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": alg["gate_up"],
                         "algorithmic_flops_per_launch": alg["gate_up_flops"],
                         "tensor_floor_us": alg["gate_up_flops"] / (tflops * 1e12) * 1e6,
                         "hbm_floor_us": alg["gate_up"] / (hbm * 1e9) * 1e6},
            "l2": "flushed before every timed step (256 MiB write)",
            "gpu_launches": KERNELS_PER_LAYER * wl.n_chunks * K,
        }
        if not args.no_cpu_baseline:
            nth = os.cpu_count() or 1
            v, secs, desc, toks, y_ref = oracle_sample(inp, wl, args.workload_cpu_budget, nth,
                                                       with_output=True)
            entry["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": nth,
                                     "kind": "oracle", "sample": "chunk 0: " + desc,
                                     "seconds": secs}
            entry["accuracy_vs_oracle"] = error_vs_oracle(layer.forward(x0, i0, w0), toks, y_ref)
        out[str(idx)] = entry
        del layer, Wg, Wu, Wd, xs_d, ids_d, w_d, y, o, xs, H, Ys, chunks, inp
        torch.cuda.empty_cache()
    return out


# ---- reference arm: the CPU oracle ------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = W.workload(args.workload)
    log(f"reference (CPU oracle): generating {wl.name} ...")
    inp = W.make_inputs(wl, seed=0)
    nth = os.cpu_count() or 1
    budget = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(inp, wl, budget, nth)
    vals, secs = [], []
    desc = ""
    for _ in range(args.steps):
        v, s, desc = oracle_sample(inp, wl, budget, nth)
        vals.append(v)
        secs.append(s)
    value = sum(v * s for v, s in zip(vals, secs)) / sum(secs)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "f": wl.f,
                   "tm": wl.tm},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nth, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def relaunch_ranks(n: int) -> int:
    """Runs this same command as n ranks under torch.distributed.run on this
    node and returns its exit code (rank 0 prints the line)."""
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node",
           str(n), "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    log(f"starting {n} ranks: {' '.join(cmd)}")
    return subprocess.run(cmd).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", type=int, default=WORKLOAD,
                    help="layer workload 1, 3, 4 or 5 (default 3, the full page-1-scale layer)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-plan-sweep", action="store_true",
                    help="skip the plan timed alone at 1M and 10M entries")
    ap.add_argument("--no-plan-gather", action="store_true",
                    help="skip the plan + gather configuration (T=2048, E=512, fp16 rows)")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the E4M3 and MXFP4 layers measured beside the bf16 one")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other layer workloads (tiny, 256-expert, long prompt)")
    ap.add_argument("--workload-cpu-budget", type=float, default=6.0,
                    help="seconds of oracle work for each other workload's cpu_baseline")
    ap.add_argument("--weights", choices=("bf16", "e4m3", "f8"), default="bf16",
                    help="expert weights: bf16 (the default measurement), E4M3 codes with "
                         "per-feature scales (bf16 activations), or f8: E4M3 weights and E4M3 "
                         "activations (both projections on 8-bit operands)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not W.workload(args.workload).ffn:
        ap.error("that workload has no expert FFN (plan + gather only)")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # N ranks were asked for without a launcher: start them, one process
        # per GPU, through torchrun on this node (rendezvous on 127.0.0.1)
        sys.exit(relaunch_ranks(args.gpus))
    rank, world, local = replicas.init_from_env(backend="nccl" if args.impl == "native" else "gloo")
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but the launcher started {world} ranks")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_native(args, rank, world, local)
    finally:
        replicas.finalize(world)


if __name__ == "__main__":
    main()
