"""GPU grouped expert GEMMs (tcgen05) vs the oracle, one stage at a time.

gate/up: H = bf16(silu(xs Wg) * (xs Wu)) against the oracle's fp64 h.
down:    Ys = bf16(w * (H Wd)) fed with the oracle's h rounded to bf16,
         against the oracle's bf16-mirror job (h rounded to bf16, fp64 down).
Inputs (plan, xs) come from the oracle.  Tolerance: max|gpu - ref| <=
1e-2 * max|ref| + 1e-3, the layer bar, applied per stage."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import dev, dev16, dev_weights, host16, inputs, layer_tolerance

pytestmark = pytest.mark.gpu


def staged_inputs(inp, E, tm):
    p = oracle.plan(inp["ids"], inp["w"], E, tm)
    xs = oracle.gather(inp["x"], p["srt_tok"])
    real = np.nonzero(p["srt_tok"] >= 0)[0]
    row_e = (np.searchsorted(p["offsets"], np.arange(p["R_pad"]), side="right") - 1).astype(np.int32)
    return p, xs, real, row_e


def to_cap(a, cap, fill=0):
    out = np.full((cap,) + a.shape[1:], fill, dtype=a.dtype)
    out[:len(a)] = a
    return out


def sample_rows(p, real, row_e, n, seed=0):
    """First and last real row of the expert with the most rows, plus the
    MMA-half and unit boundaries inside it and a random draw."""
    rng = np.random.default_rng(seed)
    big = int(np.argmax(p["counts"]))
    lo, c = int(p["offsets"][big]), int(p["counts"][big])
    picks = [lo, lo + c - 1] + [lo + r for r in (127, 128, 255, 256, 383, 384, 511, 512) if r < c]
    picks += list(rng.choice(real, size=min(n, len(real)), replace=False))
    return np.unique(np.array(picks, np.int64))


def run_case(inp, E, d, f, tm, Wg, Wu, Wd, nsample=None):
    p, xs, real, row_e = staged_inputs(inp, E, tm)
    T, k = inp["ids"].shape
    cap = B.capacity(T, k, E, tm)
    offsets = dev(p["offsets"])
    H = B.ffn_gate_up(dev16(to_cap(xs, cap)), Wg, Wu, offsets, cap)
    # the same stage reading the rows straight from x by srt_tok (TMA gather4)
    # computes the same arithmetic on the same shared-memory tiles: bit-equal
    Hr = B.ffn_gate_up_rows(dev16(inp["x"]), dev(to_cap(p["srt_tok"], cap, fill=-1)), Wg, Wu,
                            offsets, cap)
    R = p["R_pad"]
    assert torch.equal(H[:R].view(torch.int16), Hr[:R].view(torch.int16))
    rows = real if nsample is None else sample_rows(p, real, row_e, nsample)
    host = inputs_host(inp)
    h_ref, _ = oracle.expert_rows(xs, rows, row_e[rows], p["srt_w"][rows], *host)
    Hh = host16(H)
    h_gpu = W.bits_to_float(Hh[rows], "bf16").astype(np.float64)
    ok, err, bound = layer_tolerance(h_gpu, h_ref)
    assert ok, f"gate/up: max err {err} > {bound}"
    # pad rows: xs pad rows are zero, so h = silu(0) * 0 = 0 exactly
    pad = np.nonzero(p["srt_tok"] < 0)[0]
    assert np.all(Hh[pad] == 0)

    # down, fed with the oracle's h rounded to bf16 (mirror reference) on the
    # checked rows and zero rows elsewhere (rows are independent)
    hm, ysm = oracle.expert_rows(xs, rows, row_e[rows], p["srt_w"][rows], *host, mirror=True)
    Hin = np.zeros((cap, f), np.uint16)
    Hin[rows] = W.bf16_bits(hm.astype(np.float32))
    Ys = host16(B.ffn_down(dev16(Hin), Wd, offsets, dev(to_cap(p["srt_w"], cap)), cap))
    Ysh = W.bits_to_float(Ys[rows], "bf16").astype(np.float64)
    ok, err, bound = layer_tolerance(Ysh, ysm)
    assert ok, f"down: max err {err} > {bound}"
    assert np.all(Ys[pad] == 0)
    others = np.setdiff1d(np.arange(p["R_pad"]), rows)
    assert np.all((Ys[others] & 0x7FFF) == 0)   # zero H rows give +-0 rows
    return err


def inputs_host(inp):
    return inp["Wg"], inp["Wu"], inp["Wd"]


def test_ffn_tiny_all_rows():
    inp = inputs(1)
    wl = W.workload(1)
    run_case(inp, wl.E, wl.d, wl.f, wl.tm, *dev_weights(1))


@pytest.mark.parametrize("T,d,E,k,f,tm", [
    (40, 64, 3, 2, 64, 16),      # one K step, M tile half empty
    (100, 192, 5, 3, 192, 16),   # partial M tiles on both GEMMs (192 = 128 + 64)
    (300, 128, 2, 1, 256, 32),   # experts with > 128 rows: several chunks
    (257, 256, 6, 4, 704, 16),   # f = 5.5 x 128
    (64, 320, 40, 2, 128, 16),   # many experts, most with one 16-row tile
])
def test_ffn_shapes_all_rows(T, d, E, k, f, tm):
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=T + f)
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    run_case(inp, E, d, f, tm, Wg, Wu, Wd)


@pytest.mark.parametrize("d,f", [(128, 192), (64, 512)])
def test_ffn_unit_heights(d, f):
    # expert sizes on both sides of every unit-height boundary: one MMA half
    # (<= 128 rows), two halves (the second of only 16 rows, or full), and
    # experts split into a 256-row unit plus a ragged one
    counts = [16, 112, 128, 144, 240, 256, 272, 400, 528, 0, 784]
    E = len(counts)
    T = sum(counts)
    inp = W.make_layer(T, d, E, 1, f, tm=16, seed=d + f)
    ids = np.repeat(np.arange(E, dtype=np.int32), counts)
    inp["ids"] = np.random.default_rng(5).permutation(ids).reshape(T, 1)
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    run_case(inp, E, d, f, 16, Wg, Wu, Wd)


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_ffn_workloads_sampled_rows(cfg):
    wl = W.workload(cfg)
    run_case(inputs(cfg), wl.E, wl.d, wl.f, wl.tm, *dev_weights(cfg), nsample=48)


def test_ffn_deterministic():
    wl = W.workload(3)
    inp = inputs(3)
    p, xs, real, row_e = staged_inputs(inp, wl.E, wl.tm)
    cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
    args = (dev16(to_cap(xs, cap)), *dev_weights(3)[:2], dev(p["offsets"]), cap)
    a = host16(B.ffn_gate_up(*args))
    b = host16(B.ffn_gate_up(*args))
    R = p["R_pad"]
    assert np.array_equal(a[:R], b[:R])


def test_ffn_status_bad_offsets():
    # offsets not multiples of 16: that expert is skipped and flagged
    E, d, f = 2, 64, 64
    Wg = torch.zeros((E, d, f), dtype=torch.bfloat16, device="cuda")
    xs = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
    offsets = dev(np.array([0, 8, 32], np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ffn_gate_up(xs, Wg, Wg, offsets, 64, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & B.STATUS_BAD_OFFSETS


def test_ffn_wait_limit_stops_cleanly_and_reports():
    # Failure detection without a GPU fault: CTA 0's first stage waits for 16
    # bytes that never arrive, so its bounded waits run out (about 2 s), it
    # stops after letting its copies and MMAs land, and the status word says
    # so.  The other CTAs finish, and the context keeps working afterwards.
    import time
    wl = W.workload(1)
    inp = inputs(1)
    p, xs, real, row_e = staged_inputs(inp, wl.E, wl.tm)
    cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
    Wg, Wu, Wd = dev_weights(1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    B.selftest_wait_limit(dev16(to_cap(xs, cap)), Wg, Wu, dev(p["offsets"]), cap, status, cta=0)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) & B.STATUS_TIMEOUT
    assert 1.0 < elapsed < 60.0
    run_case(inp, wl.E, wl.d, wl.f, wl.tm, Wg, Wu, Wd)


@pytest.mark.parametrize("T,d,E,k,f,tm", [
    (100, 192, 5, 3, 192, 16),   # ragged M tiles on both GEMMs (192 = 128 + 64)
    (300, 128, 2, 1, 256, 32),   # experts over 128 rows
    (257, 256, 6, 4, 704, 16),   # f = 5.5 x 128
])
def test_expert_ffn_entry_point(T, d, E, k, f, tm):
    # moe_expert_ffn (gate/up and down in one call, H kept in the caller's
    # buffer) through the C ABI: H against the oracle's fp64 h, Ys against
    # the oracle's fp64 job output w * (h Wd), on every real row; pad rows 0
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=7 * T + f, skip_frac=0.1)
    p, xs, real, row_e = staged_inputs(inp, E, tm)
    cap = B.capacity(T, k, E, tm)
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    H0 = torch.full((cap, f), -7.0, dtype=torch.bfloat16, device="cuda")
    Y0 = torch.full((cap, d), -7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    H, Ys = B.expert_ffn(dev16(to_cap(xs, cap)), Wg, Wu, Wd, dev(p["offsets"]),
                         dev(to_cap(p["srt_w"], cap)), cap, H=H0, Ys=Y0, status=status)
    torch.cuda.synchronize()
    assert H.data_ptr() == H0.data_ptr() and Ys.data_ptr() == Y0.data_ptr()
    assert int(status.item()) == 0
    h_ref, ys_ref = oracle.expert_rows(xs, real, row_e[real], p["srt_w"][real], *inputs_host(inp))
    Hh, Yh = host16(H), host16(Ys)
    ok, err, bound = layer_tolerance(W.bits_to_float(Hh[real], "bf16").astype(np.float64), h_ref)
    assert ok, f"H: max err {err} > {bound}"
    ok, err, bound = layer_tolerance(W.bits_to_float(Yh[real], "bf16").astype(np.float64), ys_ref)
    assert ok, f"Ys: max err {err} > {bound}"
    pad = np.nonzero(p["srt_tok"] < 0)[0]
    assert len(pad) > 0 and np.all(Hh[pad] == 0) and np.all((Yh[pad] & 0x7FFF) == 0)
