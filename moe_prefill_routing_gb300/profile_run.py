"""A short, self-contained run of one stage for profilers (ncu).

    python -m moe_prefill_routing_gb300.profile_run --workload 3 --experts 128 \
        --stage gate_up --iters 3

Generates the named workload (optionally with fewer experts, routing redrawn
for that expert count, so that the device holds a few GB at most), runs the
whole layer once through the stage entry points, then runs the chosen stage
``--iters`` more times.  Every stage call goes through the C ABI.  With
``--weights f8`` the gather, gate/up and down stages are the E4M3-operand
ones (weights quantized on the device first; down includes the pass that
makes H's rows E4M3); with ``--weights mxfp4`` gate/up, down and the layer
run on MXFP4 weights (quantized on the device first), rows in bf16.  ``--plan-entries N`` runs the plan alone on N flat
entries (k = 10, E = 512, tm = 16, ids uniform over the experts and drawn
on the device, as in the bench's plan sweep).
"""
from __future__ import annotations

import argparse
import dataclasses
import sys

import numpy as np
import torch

from . import binding as B
from . import workload as W

STAGES = ("plan", "gather", "gate_up", "down", "combine", "layer")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--experts", type=int, default=0, help="override E (0: the workload's)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (0: the workload's)")
    ap.add_argument("--stage", choices=STAGES, default="gate_up")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--weights", choices=("bf16", "f8", "mxfp4"), default="bf16")
    ap.add_argument("--plan-entries", type=int, default=0,
                    help="run only the plan on this many uniform entries")
    a = ap.parse_args(argv)
    if a.plan_entries:
        return plan_only_run(a.plan_entries, a.iters)
    wl = W.workload(a.workload)
    if a.experts:
        wl = dataclasses.replace(wl, E=a.experts, name=f"{wl.name}_E{a.experts}")
    if a.tokens:
        wl = dataclasses.replace(wl, T=a.tokens, name=f"{wl.name}_T{a.tokens}")
    dev = torch.device("cuda", 0)
    plan_only = a.stage in ("plan", "gather")
    inp = W.make_inputs(wl, weights=not plan_only)

    def d16(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    x = d16(inp["x"])
    ids = torch.from_numpy(inp["ids"]).to(dev)
    w = torch.from_numpy(inp["w"]).to(dev)
    cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
    o = B.plan(ids, w, wl.E, wl.tm, cap=cap)
    xs = B.gather(x, o["srt_tok"], o["offsets"], wl.E, cap)
    f8 = a.weights == "f8"
    mx4 = a.weights == "mxfp4"
    if not plan_only:
        Wg, Wu, Wd = (d16(inp[n]) for n in ("Wg", "Wu", "Wd"))
        H, Ys = B.expert_ffn(xs, Wg, Wu, Wd, o["offsets"], o["srt_w"], cap)
        y = B.combine(Ys, o["pos"])
        if f8:
            Wg, Wu, Wd = (B.quantize_e4m3(t, kmajor=True) for t in (Wg, Wu, Wd))
            x8, xe = B.gather_e4m3(x, o["srt_tok"], o["offsets"], wl.E, cap)
            H8, he = B.rows_e4m3(H, o["offsets"], wl.E, cap)
        if mx4:
            Wg, Wu, Wd = (B.quantize_mxfp4(t) for t in (Wg, Wu, Wd))
    calls = {
        "plan": lambda: B.plan(ids, w, wl.E, wl.tm, cap=cap, out=o),
        "gather": lambda: B.gather(x, o["srt_tok"], o["offsets"], wl.E, cap, xs=xs),
        "gate_up": lambda: B.ffn_gate_up(xs, Wg, Wu, o["offsets"], cap, H=H),
        "down": lambda: B.ffn_down(H, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys),
        "combine": lambda: B.combine(Ys, o["pos"], y=y),
        "layer": lambda: B.layer_forward(x, ids, w, Wg, Wu, Wd, wl.tm, y=y),
    }
    if f8 and not plan_only:

        def down_f8():
            B.rows_e4m3(H, o["offsets"], wl.E, cap, H8, he)
            B.ffn_down_f8(H8, he, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys)

        calls.update({
            "gather": lambda: B.gather_e4m3(x, o["srt_tok"], o["offsets"], wl.E, cap, x8, xe),
            "gate_up": lambda: B.ffn_gate_up_f8(x8, xe, Wg, Wu, o["offsets"], cap, H=H),
            "down": down_f8,
            "layer": lambda: B.layer_forward_e4m3(x, ids, w, Wg, Wu, Wd, wl.tm, y=y,
                                                  act_e4m3=True),
        })
    if mx4 and not plan_only:
        calls.update({
            "gate_up": lambda: B.ffn_gate_up_mxfp4(xs, Wg, Wu, o["offsets"], cap, H=H),
            "down": lambda: B.ffn_down_mxfp4(H, Wd, o["offsets"], o["srt_w"], cap, Ys=Ys),
            "layer": lambda: B.layer_forward_mxfp4(x, ids, w, Wg, Wu, Wd, wl.tm, y=y),
        })
    for _ in range(a.iters):
        calls[a.stage]()
    torch.cuda.synchronize(dev)
    flat = inp["ids"].ravel()
    counts = np.bincount(flat[flat >= 0], minlength=wl.E)
    print(f"{wl.name}: stage {a.stage} x{a.iters}; active experts {(counts > 0).sum()}, "
          f"R_pad {int((-(-counts // wl.tm) * wl.tm).sum())}", file=sys.stderr)


def plan_only_run(n: int, iters: int):
    k, E, tm = 10, 512, 16
    T = n // k
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(1234 + n)
    ids = torch.randint(0, E, (T, k), generator=gen, device=dev, dtype=torch.int32)
    w = torch.rand((T, k), generator=gen, device=dev)
    cap = B.capacity(T, k, E, tm)
    o = B.plan(ids, w, E, tm, cap=cap)
    for _ in range(iters):
        B.plan(ids, w, E, tm, cap=cap, out=o)
    torch.cuda.synchronize(dev)
    print(f"plan of {T * k} uniform entries (E={E}, k={k}) x{iters + 1}; "
          f"R_pad {int(o['offsets'][-1])}", file=sys.stderr)


if __name__ == "__main__":
    main()
