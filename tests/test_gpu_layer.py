"""moe_layer_forward (plan -> gather -> gate/up -> down -> combine in one call)
vs the oracle: max|y - ref| <= 1e-2 * max|ref| + 1e-3, bf16 operands with
fp32 accumulation.  Full outputs on small shapes and on the full-size
layers (the first chunk of the long prompt included), in the same launch
configuration the benchmark times; on the other long-prompt chunks, sampled
tokens that the oracle computes one by one.  The plan and the gathered rows left in the
workspace are also checked bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import (dev, dev16, dev_weights, host16, host_f, inputs, layer_tolerance, rel_l2,
                     sample_tokens)

pytestmark = pytest.mark.gpu


def run_layer(inp, Wg, Wu, Wd, tm):
    T, d = inp["x"].shape
    k = inp["ids"].shape[1]
    E, _, f = Wg.shape
    ws = torch.empty(B.workspace_bytes(T, d, E, k, f, tm), dtype=torch.uint8, device="cuda")
    y = B.layer_forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]), Wg, Wu, Wd, tm, ws=ws)
    torch.cuda.synchronize()
    return y, ws


def ws_view(ws, L, field, dtype, n):
    b = ws[L[field]:L[field] + n * torch.tensor([], dtype=dtype).element_size()]
    return b.view(dtype)


def check_workspace_plan(ws, inp, E, d, f, tm):
    T, k = inp["ids"].shape
    L = B.workspace_layout(T, d, E, k, f, tm)
    ref = oracle.plan(inp["ids"], inp["w"], E, tm)
    R = ref["R_pad"]
    assert ws_view(ws, L, "offsets", torch.int32, E + 1).cpu().numpy().tolist() == ref["offsets"].tolist()
    assert np.array_equal(ws_view(ws, L, "srt_tok", torch.int32, R).cpu().numpy(), ref["srt_tok"])
    assert np.array_equal(ws_view(ws, L, "srt_w", torch.int32, R).cpu().numpy(),
                          ref["srt_w"].view(np.int32))
    assert np.array_equal(ws_view(ws, L, "pos", torch.int32, T * k).cpu().numpy().reshape(T, k),
                          ref["pos"])
    xs = host16(ws_view(ws, L, "xs", torch.int16, R * d).view(R, d))
    assert np.array_equal(xs, oracle.gather(inp["x"], ref["srt_tok"]))
    assert B.read_status(ws) == 0


def test_layer_tiny_full_output():
    wl = W.workload(1)
    inp = inputs(1)
    y, ws = run_layer(inp, *dev_weights(1), wl.tm)
    got = host_f(y)
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    ok, err, bound = layer_tolerance(got, ref)
    assert ok, (err, bound)
    mirror = oracle.layer(inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"], mirror=True)
    print(f"tiny layer: max err {err:.3e} (bound {bound:.3e}); rel-L2 vs fp64 {rel_l2(got, ref):.3e}, "
          f"vs bf16 mirror {rel_l2(got, mirror):.3e}")
    check_workspace_plan(ws, inp, wl.E, wl.d, wl.f, wl.tm)


@pytest.mark.parametrize("T,d,E,k,f,tm,skip", [
    (50, 64, 4, 2, 64, 16, 0.0),
    (123, 192, 9, 3, 192, 16, 0.2),      # ragged M tiles, skipped slots
    (64, 256, 3, 3, 128, 32, 0.0),       # tm = 32, experts over 128 rows
    (200, 128, 70, 4, 704, 16, 0.1),     # f = 5.5 x 128
    (1, 128, 8, 8, 64, 16, 0.0),         # one token
    (300, 128, 4096, 4, 64, 16, 0.0),    # E at its limit: largest GEMM shared-memory table
    (9000, 64, 64, 8, 64, 16, 0.05),     # T*k above 16 x 4096: the multi-kernel plan
])
def test_layer_shapes_full_output(T, d, E, k, f, tm, skip):
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=3 * T + E, skip_frac=skip)
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    y, ws = run_layer(inp, Wg, Wu, Wd, tm)
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    ok, err, bound = layer_tolerance(host_f(y), ref)
    assert ok, (err, bound)
    check_workspace_plan(ws, inp, E, d, f, tm)


@pytest.mark.parametrize("cfg,chunk", [(3, 0), (4, 0), (5, 0)])
def test_layer_workloads_full_output(cfg, chunk):
    # every token of the full-size layers (the full page-1-scale layer, the
    # 256-expert layer, the first chunk of the long prompt), in the launch
    # configuration the benchmark times, against the oracle run on all tokens
    wl = W.workload(cfg)
    inp = inputs(cfg)
    y, ws = run_layer(inp, *dev_weights(cfg), wl.tm)
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    got = host_f(y)
    assert got.shape == ref.shape == (wl.T, wl.d)
    ok, err, bound = layer_tolerance(got, ref)
    assert ok, (err, bound)
    assert B.read_status(ws) == 0
    print(f"cfg {cfg} chunk {chunk}: all {wl.T} tokens, max err {err:.3e} (bound {bound:.3e}), "
          f"rel-L2 {rel_l2(got, ref):.3e}")


@pytest.mark.parametrize("cfg,chunk", [(5, 5)])
def test_layer_workloads_sampled_tokens(cfg, chunk):
    # the other chunks of the long prompt: tokens the oracle computes one by one
    wl = W.workload(cfg)
    inp = W.make_inputs(cfg, chunk=chunk, weights=False)
    host_w = inputs(cfg)
    y, ws = run_layer(inp, *dev_weights(cfg), wl.tm)
    toks = sample_tokens(inp["ids"], 40, seed=cfg)
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], host_w["Wg"], host_w["Wu"], host_w["Wd"],
                       tokens=toks)
    got = host_f(y)[toks]
    ok, err, bound = layer_tolerance(got, ref)
    assert ok, (err, bound)
    assert B.read_status(ws) == 0
    print(f"cfg {cfg} chunk {chunk}: {len(toks)} tokens, max err {err:.3e} (bound {bound:.3e}), "
          f"rel-L2 {rel_l2(got, ref):.3e}")


def test_layer_full_size_plan_and_gather_in_workspace():
    wl = W.workload(3)
    inp = inputs(3)
    _, ws = run_layer(inp, *dev_weights(3), wl.tm)
    check_workspace_plan(ws, inp, wl.E, wl.d, wl.f, wl.tm)


def test_layer_deterministic():
    wl = W.workload(3)
    inp = inputs(3)
    a, _ = run_layer(inp, *dev_weights(3), wl.tm)
    b, _ = run_layer(inp, *dev_weights(3), wl.tm)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layer_all_slots_skipped_gives_zero():
    inp = W.make_layer(20, 64, 4, 2, 64, seed=1)
    inp["ids"][:] = -1
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    y, ws = run_layer(inp, Wg, Wu, Wd, 16)
    assert torch.all(y.float() == 0)


def test_layer_moe_layer_host_path():
    wl = W.workload(1)
    inp = inputs(1)
    layer = B.MoeLayer(*dev_weights(1), tm=wl.tm)
    x_h = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_h = torch.from_numpy(inp["ids"]).pin_memory()
    w_h = torch.from_numpy(inp["w"]).pin_memory()
    y_h = torch.empty((wl.T, wl.d), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(x_h, ids_h, w_h, y_h)
    torch.cuda.synchronize()
    y, _ = run_layer(inp, *dev_weights(1), wl.tm)
    assert torch.equal(y_h.view(torch.int16), y.cpu().view(torch.int16))


def host_chunks(chunks, d):
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    xs = [torch.from_numpy(c["x"].view(np.int16)).view(torch.bfloat16).pin_memory() for c in chunks]
    ids = [pin(c["ids"]) for c in chunks]
    ws = [pin(c["w"]) for c in chunks]
    ys = [torch.full((c["x"].shape[0], d), float("nan"), dtype=torch.bfloat16).pin_memory()
          for c in chunks]
    return xs, ids, ws, ys


@pytest.mark.parametrize("n_chunks", [1, 2, 3, 6])
def test_prefill_host_chunks(n_chunks):
    # a prompt as n chunks in host memory: every chunk's y equals the device
    # layer's bit for bit and meets the oracle's bar
    T, d, E, k, f, tm = 300, 256, 16, 4, 192, 16
    chunks = [W.make_layer(T, d, E, k, f, tm=tm, seed=40 + c, skip_frac=0.05)
              for c in range(n_chunks)]
    Wg, Wu, Wd = (dev16(chunks[0][n]) for n in ("Wg", "Wu", "Wd"))
    layer = B.MoeLayer(Wg, Wu, Wd, tm=tm)
    xs, ids, ws, ys = host_chunks(chunks, d)
    layer.forward_host_chunks(xs, ids, ws, ys)
    torch.cuda.synchronize()
    assert B.read_status(layer._host_ws) == 0
    for c, inp in enumerate(chunks):
        ref_dev = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
        torch.cuda.synchronize()
        assert torch.equal(ys[c].view(torch.int16), ref_dev.cpu().view(torch.int16)), c
        ref = oracle.layer(inp["x"], inp["ids"], inp["w"], chunks[0]["Wg"], chunks[0]["Wu"],
                           chunks[0]["Wd"])
        ok, err, bound = layer_tolerance(host_f(ys[c]), ref)
        assert ok, (c, err, bound)


def test_prefill_host_chunks_shared_buffers():
    # the same input chunk five times into one output buffer: it holds that
    # chunk's y; a later call on the same layer reuses the workspace
    T, d, E, k, f, tm = 64, 128, 8, 2, 128, 16
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=7)
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = B.MoeLayer(Wg, Wu, Wd, tm=tm)
    xs, ids, ws, ys = host_chunks([inp], d)
    layer.forward_host_chunks(xs * 5, ids * 5, ws * 5, ys * 5)
    torch.cuda.synchronize()
    ref = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])).cpu()
    assert torch.equal(ys[0].view(torch.int16), ref.view(torch.int16))
    other = W.make_layer(T, d, E, k, f, tm=tm, seed=8)
    xs2, ids2, ws2, ys2 = host_chunks([other], d)
    layer.forward_host_chunks(xs2, ids2, ws2, ys2)
    torch.cuda.synchronize()
    ref2 = layer.forward(dev16(other["x"]), dev(other["ids"]), dev(other["w"])).cpu()
    assert torch.equal(ys2[0].view(torch.int16), ref2.view(torch.int16))


def test_prefill_host_long_prompt_chunks_sampled():
    # the long-prompt workload's chunks through the host path, two of them,
    # sampled tokens against the oracle
    wl = W.workload(5)
    host_w = inputs(5)
    chunks = [W.make_inputs(wl, chunk=c, weights=False) for c in (0, 1)]
    layer = B.MoeLayer(*dev_weights(5), tm=wl.tm)
    xs, ids, ws, ys = host_chunks(chunks, wl.d)
    layer.forward_host_chunks(xs, ids, ws, ys)
    torch.cuda.synchronize()
    assert B.read_status(layer._host_ws) == 0
    for c, inp in enumerate(chunks):
        toks = sample_tokens(inp["ids"], 24, seed=c)
        ref = oracle.layer(inp["x"], inp["ids"], inp["w"], host_w["Wg"], host_w["Wu"],
                           host_w["Wd"], tokens=toks)
        ok, err, bound = layer_tolerance(host_f(ys[c])[toks], ref)
        assert ok, (c, err, bound)
