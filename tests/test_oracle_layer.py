"""Pins of the oracle's expert FFN, combine and 16-bit conversions (CPU only).

The layer follows the flat job pass of "Batched resident MoE experts on Apple
Silicon: a flat parallel expert pass" (section 1: per job gate/up projection,
gated activation, weighted down projection; section 3: per-token top-k
summation order).  Pins: a hand-worked fixture, a pure-Python dense per-token
evaluation that must agree bit for bit, closed forms, and dense numpy/scipy
cross-checks for cases that reduce to a plain SwiGLU MLP.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from moe_prefill_routing_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def widen(bits, dtype="bf16"):
    return W.bits_to_float(bits, dtype).astype(np.float64)


def brute_layer(x, ids, w, Wg, Wu, Wd, x_dtype="bf16"):
    """Each token run densely through its k experts, with Python floats in
    the order the definition states (sum over c, then over n, then over j)."""
    T, d = x.shape
    k = ids.shape[1]
    E, _, f = Wg.shape
    xv = widen(x, x_dtype).tolist()
    g_w, u_w, d_w = widen(Wg).tolist(), widen(Wu).tolist(), widen(Wd).tolist()
    y = []
    for t in range(T):
        yt = [0.0] * d
        for j in range(k):
            e = int(ids[t, j])
            if e == -1:
                continue
            g = [0.0] * f
            u = [0.0] * f
            for c in range(d):
                for n in range(f):
                    g[n] += xv[t][c] * g_w[e][c][n]
                    u[n] += xv[t][c] * u_w[e][c][n]
            h = [g[n] / (1.0 + math.exp(-g[n])) * u[n] for n in range(f)]
            o = [0.0] * d
            for n in range(f):
                for m in range(d):
                    o[m] += h[n] * d_w[e][n][m]
            wt = float(np.float32(w[t, j]))
            for m in range(d):
                yt[m] += wt * o[m]
        y.append(yt)
    return np.array(y, np.float64)


def test_layer_hand_worked():
    v = {}
    for line in open(os.path.join(GOLDEN, "layer_worked_example.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            key, *vals = line.split()
            v[key] = vals
    T, d, f, E, k = (int(v[n][0]) for n in ("T", "d", "f", "E", "k"))
    x = W.bf16_bits(np.array(v["x"], np.float32).reshape(T, d))
    ids = np.array(v["ids"], np.int32).reshape(T, k)
    w = np.array(v["w"], np.float32).reshape(T, k)
    Wg = W.bf16_bits(np.array(v["Wg"], np.float32).reshape(E, d, f))
    Wu = W.bf16_bits(np.array(v["Wu"], np.float32).reshape(E, d, f))
    Wd = W.bf16_bits(np.array(v["Wd"], np.float32).reshape(E, f, d))
    y = oracle.layer(x, ids, w, Wg, Wu, Wd)
    want = np.array(v["y"], np.float64).reshape(T, d)
    np.testing.assert_allclose(y, want, rtol=4e-16, atol=0)
    # the closed form the fixture was worked from: s = silu(1) = e / (1 + e)
    s = math.e / (1.0 + math.e)
    np.testing.assert_allclose(want, [[2 * s, -0.5 * s]], rtol=4e-16)


@pytest.mark.parametrize("seed", range(6))
def test_layer_vs_brute_force_bit_identical(seed):
    rng = np.random.default_rng(100 + seed)
    T, d, E, k, f = (int(rng.integers(1, 6)), int(rng.integers(1, 17)), int(rng.integers(1, 7)),
                     int(rng.integers(1, 4)), int(rng.integers(1, 9)))
    x_dtype = "f16" if seed % 3 == 2 else "bf16"
    conv = W.f16_bits if x_dtype == "f16" else W.bf16_bits
    x = conv(rng.standard_normal((T, d)).astype(np.float32))
    Wg = W.bf16_bits(0.5 * rng.standard_normal((E, d, f)).astype(np.float32))
    Wu = W.bf16_bits(0.5 * rng.standard_normal((E, d, f)).astype(np.float32))
    Wd = W.bf16_bits(0.5 * rng.standard_normal((E, f, d)).astype(np.float32))
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y = oracle.layer(x, ids, w, Wg, Wu, Wd, x_dtype=x_dtype, nthreads=3)
    yb = brute_layer(x, ids, w, Wg, Wu, Wd, x_dtype=x_dtype)
    assert np.array_equal(y.view(np.uint64), yb.view(np.uint64))


def test_single_job_closed_form():
    # d = f = 1: y = w * silu(a * xg) * (b * xu) * c with a library sigmoid
    for a, b, c, xv, wt in [(1.5, -0.75, 2.0, 1.0, 0.5), (-3.0, 0.25, -1.0, 2.0, 0.125),
                            (0.0, 4.0, 1.0, 1.0, 1.0), (20.0, 1.0, 1.0, 1.0, 1.0)]:
        x = W.bf16_bits(np.array([[xv]], np.float32))
        Wg = W.bf16_bits(np.array([[[a]]], np.float32))
        Wu = W.bf16_bits(np.array([[[b]]], np.float32))
        Wd = W.bf16_bits(np.array([[[c]]], np.float32))
        y = oracle.layer(x, np.zeros((1, 1), np.int32), np.array([[wt]], np.float32), Wg, Wu, Wd)
        g, u = a * xv, b * xv
        want = wt * (g * expit(g)) * u * c
        np.testing.assert_allclose(y[0, 0], want, rtol=1e-15, atol=1e-300)


@pytest.mark.parametrize("x_dtype", ["bf16", "f16"])
def test_single_expert_is_dense_swiglu_mlp(x_dtype):
    # E = 1, k = 1, w = 1: the layer is silu(X Wg) * (X Wu) then Wd, which a
    # float64 BLAS computes in its own order
    rng = np.random.default_rng(7)
    T, d, f = 11, 40, 24
    conv = W.f16_bits if x_dtype == "f16" else W.bf16_bits
    x = conv(rng.standard_normal((T, d)).astype(np.float32))
    Wg = W.bf16_bits(0.2 * rng.standard_normal((1, d, f)).astype(np.float32))
    Wu = W.bf16_bits(0.2 * rng.standard_normal((1, d, f)).astype(np.float32))
    Wd = W.bf16_bits(0.2 * rng.standard_normal((1, f, d)).astype(np.float32))
    y = oracle.layer(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32), Wg, Wu, Wd,
                     x_dtype=x_dtype)
    X = widen(x, x_dtype)
    G, U = X @ widen(Wg)[0], X @ widen(Wu)[0]
    ref = (G * expit(G) * U) @ widen(Wd)[0]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_routed_layer_is_weighted_sum_of_expert_mlps():
    # every token, every slot: w * MLP_e(x) summed over slots, via numpy
    inp = W.make_inputs(1)
    y = oracle.layer(inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    X = widen(inp["x"])
    G = np.einsum("tc,ecn->etn", X, widen(inp["Wg"]))
    U = np.einsum("tc,ecn->etn", X, widen(inp["Wu"]))
    O = np.einsum("etn,enm->etm", G * expit(G) * U, widen(inp["Wd"]))
    ids, w = inp["ids"], inp["w"].astype(np.float64)
    ref = sum(w[:, j, None] * O[ids[:, j], np.arange(ids.shape[0])] for j in range(ids.shape[1]))
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-13)


def test_token_subset_and_threads_do_not_change_results():
    inp = W.make_inputs(1)
    args = (inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    full = oracle.layer(*args, nthreads=1)
    toks = np.array([63, 0, 17, 17, 5], np.int32)
    sub = oracle.layer(*args, tokens=toks, nthreads=4)
    assert np.array_equal(sub, full[toks])


def test_expert_rows_and_combine_rebuild_the_layer():
    # stage views: plan -> gather -> per-row (h, w*o) -> combine of rows in slot order
    inp = W.make_inputs(1)
    wl = W.workload(1)
    p = oracle.plan(inp["ids"], inp["w"], wl.E, wl.tm)
    xs = oracle.gather(inp["x"], p["srt_tok"])
    real = np.nonzero(p["srt_tok"] >= 0)[0]
    row_e = np.searchsorted(p["offsets"], real, side="right").astype(np.int32) - 1
    h, ys = oracle.expert_rows(xs, real, row_e, p["srt_w"][real], inp["Wg"], inp["Wu"], inp["Wd"])
    y = oracle.layer(*(inp[n] for n in ("x", "ids", "w", "Wg", "Wu", "Wd")))
    # rebuild y from the per-row results, slot order, fp64
    row_of = {int(r): i for i, r in enumerate(real)}
    yr = np.zeros_like(y)
    for t in range(wl.T):
        for j in range(wl.k):
            yr[t] += ys[row_of[int(p["pos"][t, j])]]
    assert np.array_equal(yr, y)
    # oracle.combine over bf16 rows equals the same slot-ordered sum
    Ys = W.bf16_bits(np.zeros((p["R_pad"], wl.d), np.float32))
    Ys[real] = W.bf16_bits(ys.astype(np.float32))
    yc = oracle.combine(Ys, p["pos"])
    want = np.zeros_like(y)
    for j in range(wl.k):
        want += widen(Ys)[p["pos"][:, j]]
    assert np.array_equal(yc, want)


def test_mirror_reference_is_close_to_exact():
    inp = W.make_inputs(1)
    args = (inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"])
    y = oracle.layer(*args)
    ym = oracle.layer(*args, mirror=True)
    rel = np.linalg.norm(ym - y) / np.linalg.norm(y)
    assert 0 < rel < 1e-2
    # mirror outputs are bf16 values
    assert np.array_equal(ym, widen(W.bf16_bits(ym.astype(np.float32))))


def test_value16_matches_library_widening():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref_f16 = allbits.view(np.float16).astype(np.float64)
    ref_bf16 = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b in list(range(0, 65536, 97)) + [0x0001, 0x03FF, 0x0400, 0x7BFF, 0x8001, 0xFBFF, 0x7C00]:
        for dtype, ref in (("f16", ref_f16), ("bf16", ref_bf16)):
            got = oracle.value16(b, dtype)
            if np.isnan(ref[b]):
                assert math.isnan(got)
            else:
                assert got == ref[b], (dtype, hex(b))


def test_round_bf16_matches_library_rounding():
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                           [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0, 1e-40]])
    ref = torch.from_numpy(vals).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(v) for v in vals])
    assert np.array_equal(got, ref)
