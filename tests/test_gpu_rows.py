"""GPU gather (bit-exact) and combine (fp32 slot-ordered sum) vs the oracle.

Inputs to each stage come from the oracle's own plan, so a stage is checked
on its own."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import dev, dev16, host16, inputs

pytestmark = pytest.mark.gpu

POISON16 = 0x7BAD


def gpu_gather(x_bits, x_dtype, plan, E, cap):
    dt = torch.float16 if x_dtype == "f16" else torch.bfloat16
    x = dev16(x_bits, dt)
    srt_tok = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    srt_tok[:plan["R_pad"]] = dev(plan["srt_tok"])
    xs = torch.full((cap, x.shape[1]), POISON16, dtype=torch.int16, device="cuda").view(dt)
    B.gather(x, srt_tok, dev(plan["offsets"]), E, cap, xs=xs)
    return host16(xs)


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_gather_workloads_bit_exact(cfg):
    wl = W.workload(cfg)
    inp = inputs(cfg) if cfg != 3 else W.make_inputs(3, weights=False)
    p = oracle.plan(inp["ids"], inp["w"], wl.E, wl.tm)
    cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
    xs = gpu_gather(inp["x"], wl.x_dtype, p, wl.E, cap)
    R = p["R_pad"]
    assert np.array_equal(xs[:R], oracle.gather(inp["x"], p["srt_tok"]))
    assert np.all(xs[R:] == POISON16)          # rows past R_pad untouched


@pytest.mark.parametrize("T,d,E,k,tm", [(1, 8, 1, 1, 16), (33, 24, 5, 3, 16), (129, 136, 7, 2, 32),
                                        (300, 2816, 128, 8, 16), (50, 4096, 9, 4, 64)])
def test_gather_edges_bit_exact(T, d, E, k, tm):
    inp = W.make_layer(T, d, E, k, 0, tm=tm, seed=T + d, skip_frac=0.1, weights=False)
    p = oracle.plan(inp["ids"], inp["w"], E, tm)
    cap = B.capacity(T, k, E, tm)
    xs = gpu_gather(inp["x"], "bf16", p, E, cap)
    assert np.array_equal(xs[:p["R_pad"]], oracle.gather(inp["x"], p["srt_tok"]))


def combine_bound(Ys_bits, pos, ref):
    """|gpu - ref| allowed: one bf16 rounding of the result (2^-9 relative,
    taken as 2^-8) plus k fp32 roundings of the running sum."""
    k = pos.shape[1]
    absum = oracle.combine(W.bf16_bits(np.abs(W.bits_to_float(Ys_bits, "bf16"))), pos)
    return 2.0 ** -8 * np.abs(ref) + k * 2.0 ** -23 * absum + 1e-37


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_combine_vs_oracle(cfg):
    wl = W.workload(cfg)
    inp = W.make_inputs(cfg, weights=False)
    p = oracle.plan(inp["ids"], inp["w"], wl.E, wl.tm)
    rng = np.random.default_rng(cfg)
    Ys = W.bf16_bits(0.1 * rng.standard_normal((p["R_pad"], wl.d)).astype(np.float32))
    y = B.combine(dev16(Ys), dev(p["pos"]))
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle.combine(Ys, p["pos"])
    assert np.all(np.abs(got - ref) <= combine_bound(Ys, p["pos"], ref))


def test_combine_skipped_slots_and_ragged_d():
    T, k, d = 77, 5, 200
    rng = np.random.default_rng(9)
    Ys = W.bf16_bits(rng.standard_normal((300, d)).astype(np.float32))
    pos = rng.integers(0, 300, size=(T, k)).astype(np.int32)
    pos[rng.random((T, k)) < 0.25] = -1
    pos[5] = -1                                   # a token with every slot skipped -> 0
    got = B.combine(dev16(Ys), dev(pos)).float().cpu().numpy().astype(np.float64)
    ref = oracle.combine(Ys, pos)
    assert np.all(got[5] == 0)
    assert np.all(np.abs(got - ref) <= combine_bound(Ys, pos, ref))


def test_combine_order_is_slot_order():
    # slots 2^24, 1, -2^24: summed from zero in slot order, fp32 gives
    # (2^24 + 1) -> 2^24 (tie to even), then 0; any other order gives 1
    d = 8
    rows = np.array([[2.0 ** 24] * d, [1.0] * d, [-(2.0 ** 24)] * d], np.float32)
    Ys = W.bf16_bits(rows)
    got = B.combine(dev16(Ys), dev(np.array([[0, 1, 2]], np.int32))).float().cpu().numpy()
    assert np.all(got == 0.0)
    got = B.combine(dev16(Ys), dev(np.array([[0, 2, 1]], np.int32))).float().cpu().numpy()
    assert np.all(got == 1.0)


def test_combine_order_across_slot_groups():
    # the combine copies slot rows in groups of four; the sum still runs in
    # slot order across the groups: 2^24 (slot 0) + 1 (slot 4) -> 2^24 (tie
    # to even), then - 2^24 (slot 8) -> 0; any other order gives 1
    d = 8
    rows = np.array([[2.0 ** 24] * d, [1.0] * d, [-(2.0 ** 24)] * d, [0.0] * d], np.float32)
    Ys = W.bf16_bits(rows)
    pos = np.array([[0, 3, 3, 3, 1, 3, -1, 3, 2]], np.int32)
    got = B.combine(dev16(Ys), dev(pos)).float().cpu().numpy()
    assert np.all(got == 0.0)
    pos = np.array([[0, 3, 3, 3, 2, 3, -1, 3, 1]], np.int32)
    got = B.combine(dev16(Ys), dev(pos)).float().cpu().numpy()
    assert np.all(got == 1.0)


def test_combine_many_slots_several_segments():
    # k = 37 (ten groups of slots, more slots than lanes), d = 808: three
    # full 256-column segments and a ragged one of 40 columns
    T, k, d = 50, 37, 808
    rng = np.random.default_rng(12)
    Ys = W.bf16_bits(rng.standard_normal((600, d)).astype(np.float32))
    pos = rng.integers(0, 600, size=(T, k)).astype(np.int32)
    pos[rng.random((T, k)) < 0.2] = -1
    got = B.combine(dev16(Ys), dev(pos)).float().cpu().numpy().astype(np.float64)
    ref = oracle.combine(Ys, pos)
    assert np.all(np.abs(got - ref) <= combine_bound(Ys, pos, ref))
