"""Pins of the oracle's E4M3 expert weights (CPU).

The codec is checked against torch's float8_e4m3fn (a library implementation
of the same OCP format) and against the format's closed-form values; the
quantizer against its error bound and the properties its definition fixes;
the layer with E4M3 weights against the bf16 layer (itself pinned by the
other oracle tests) on weights that both forms represent exactly, and
against a dense float64 MLP for a single expert."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import workload as W

pytestmark = pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="no float8 in torch")


def torch_decode(codes):
    return torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def torch_encode(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_all_codes_matches_torch():
    codes = np.arange(256)
    ours = np.array([oracle.e4m3_value(c) for c in codes])
    ref = torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_closed_forms():
    assert oracle.e4m3_value(0x7E) == 448.0            # largest finite
    assert oracle.e4m3_value(0x01) == 2.0 ** -9        # smallest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6        # smallest normal
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xB8) == -1.0
    # the finite magnitudes increase with the code
    mags = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(mags, mags[1:]))


def test_encode_matches_torch_inside_range():
    rng = np.random.default_rng(0)
    mags = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (mags[:-1] + mags[1:]) / 2            # every tie
    vals = np.concatenate([
        mags, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 0.01,
        rng.standard_normal(5000) * 1e-4,
    ]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    vals = vals[np.abs(vals) <= 448]
    ours = np.array([oracle.e4m3_encode(v) for v in vals], np.uint8)
    assert np.array_equal(ours, torch_encode(vals))


def test_encode_saturates_and_keeps_sign():
    for v, code in ((448.0, 0x7E), (449.0, 0x7E), (1e30, 0x7E), (-500.0, 0xFE),
                    (-0.0, 0x80), (0.0, 0x00), (-(2.0 ** -11), 0x80)):
        assert oracle.e4m3_encode(v) == code, v


def test_quantize_definition_properties():
    rng = np.random.default_rng(1)
    E, K, M = 3, 40, 24
    Wf = (rng.standard_normal((E, K, M)) * 0.02).astype(np.float32)
    Wf[1, :, 5] = 0.0                                  # an all-zero column
    Wf[2, :, 7] = 0.0
    Wf[2, 3, 7] = -3e-3                                # one non-zero entry
    Wb = W.bf16_bits(Wf)
    Wv = W.bits_to_float(Wb, "bf16").astype(np.float64)
    q, s = oracle.quantize_e4m3(Wb)
    assert q.shape == (E, K, M) and s.shape == (E, M)
    amax = np.abs(Wv).max(axis=1)
    assert s[1, 5] == 1.0 and np.all(q[1, :, 5] == 0)
    # scale is amax/448 in fp32; the largest entry of each column becomes +-448
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz].astype(np.float32) / np.float32(448.0))[...])
    for e in range(E):
        for m in range(M):
            if amax[e, m] == 0:
                continue
            kmax = int(np.argmax(np.abs(Wv[e, :, m])))
            assert q[e, kmax, m] & 0x7F == 0x7E
    # codes are the nearest E4M3 values of W / scale (torch rounds the same way)
    ratio = (Wv.astype(np.float32) / s[:, None, :]).astype(np.float32)
    assert np.array_equal(q, torch_encode(ratio.ravel()).reshape(q.shape))
    # error bound: half a step of the E4M3 grid, times the scale
    # (the fp32 division W / scale adds at most 2^-24 relative before rounding)
    deq = oracle.dequantize_e4m3(q, s)
    sb = np.broadcast_to(s[:, None, :].astype(np.float64), Wv.shape)
    err = np.abs(deq - Wv)
    normal = np.abs(Wv) >= (2.0 ** -6) * sb
    assert np.all(err[normal] <= (2.0 ** -4) * (1 + 2.0 ** -20) * np.abs(Wv)[normal])
    assert np.all(err[~normal] <= (2.0 ** -10) * (1 + 2.0 ** -20) * sb[~normal])


def pow2_weights(E, K, M, seed):
    """E4M3 codes with power-of-two scales: the dequantized weights are
    exact in bf16, so the bf16 path sees the same values."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(E, K, M)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38                          # no NaN codes
    s = (2.0 ** rng.integers(-9, -4, size=(E, M))).astype(np.float32)
    deq = oracle.dequantize_e4m3(q, s)
    bits = W.bf16_bits(deq.astype(np.float32))
    assert np.array_equal(W.bits_to_float(bits, "bf16").astype(np.float64), deq)
    return (q, s), bits


@pytest.mark.parametrize("mirror", [False, True])
def test_layer_e4m3_equals_bf16_on_exact_weights(mirror):
    T, d, E, k, f = 12, 64, 4, 2, 32
    inp = W.make_layer(T, d, E, k, f, seed=3, weights=False)
    g8, gb = pow2_weights(E, d, f, 1)
    u8, ub = pow2_weights(E, d, f, 2)
    d8, db = pow2_weights(E, f, d, 3)
    y8 = oracle.layer(inp["x"], inp["ids"], inp["w"], g8, u8, d8, mirror=mirror)
    yb = oracle.layer(inp["x"], inp["ids"], inp["w"], gb, ub, db, mirror=mirror)
    assert np.array_equal(y8, yb)
    rows = np.arange(5, dtype=np.int64)
    re = np.array([0, 1, 2, 3, 1], np.int32)
    rw = np.ones(5, np.float32)
    xs = inp["x"][:5]
    h8, ys8 = oracle.expert_rows(xs, rows, re, rw, g8, u8, d8, mirror=mirror)
    hb, ysb = oracle.expert_rows(xs, rows, re, rw, gb, ub, db, mirror=mirror)
    assert np.array_equal(h8, hb) and np.array_equal(ys8, ysb)


def test_layer_e4m3_single_expert_dense_mlp():
    # E = 1, k = 1, w = 1: y = (silu(x Wg) * (x Wu)) Wd with the dequantized
    # weights, in float64 numpy
    T, d, f = 9, 32, 16
    inp = W.make_layer(T, d, 1, 1, f, seed=4)
    inp["w"][:] = 1.0
    q = [oracle.quantize_e4m3(inp[n]) for n in ("Wg", "Wu", "Wd")]
    Wg, Wu, Wd = (oracle.dequantize_e4m3(*p)[0] for p in q)
    x = W.bits_to_float(inp["x"], "bf16").astype(np.float64)
    g, u = x @ Wg, x @ Wu
    ref = (g / (1.0 + np.exp(-g)) * u) @ Wd
    y = oracle.layer(inp["x"], inp["ids"], inp["w"], *q)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_row_quantize_scale_is_the_smallest_power_of_two():
    rng = np.random.default_rng(7)
    rows = [rng.standard_normal(40) * 10.0 ** p for p in (-30, -8, -2, 0, 1, 2, 3, 5, 30)]
    rows += [np.zeros(40), np.full(40, 448.0), np.full(40, 449.0), np.full(40, 224.0),
             np.array([448.0 * 2 ** 5] + [1.0] * 39)]
    x = W.bf16_bits(np.array(rows, np.float32))
    xv = W.bits_to_float(x, "bf16").astype(np.float64)
    q, e = oracle.quantize_rows_e4m3(x)
    for r in range(len(rows)):
        amax = np.abs(xv[r]).max()
        if amax == 0:
            assert e[r] == 0 and np.all(q[r] & 0x7F == 0)
            continue
        assert amax <= 448.0 * 2.0 ** e[r]                 # fits
        assert amax > 448.0 * 2.0 ** (e[r] - 1)            # and is the smallest that does
        scaled = (xv[r] * 2.0 ** -int(e[r])).astype(np.float32)
        assert np.array_equal(q[r], torch_encode(scaled))  # nearest codes, ties to even


def rows_e4m3_torch(v):
    """The per-row rule restated with torch's encoder: e the smallest integer
    with max|row| <= 448 * 2^e, values decode(encode(row * 2^-e)) * 2^e."""
    out = np.zeros_like(v)
    for r in range(v.shape[0]):
        amax = np.abs(v[r]).max()
        e = 0
        if amax > 0:
            e = int(np.floor(np.log2(amax))) - 8
            while amax > 448.0 * 2.0 ** e:
                e += 1
            while amax <= 448.0 * 2.0 ** (e - 1):
                e -= 1
        codes = torch_encode((v[r] * 2.0 ** -e).astype(np.float32))
        out[r] = torch_decode(codes) * 2.0 ** e
    return out


@pytest.mark.parametrize("mirror", [False, True])
def test_layer_e4m3_activations_dense_reference(mirror):
    # E = 1, k = 1, w = 1: gate/up on the x rows' E4M3 values, down on the
    # E4M3 values of h (rounded to bf16 first in the mirror), in float64
    # numpy with torch's E4M3 rounding
    T, d, f = 12, 64, 32
    inp = W.make_layer(T, d, 1, 1, f, seed=11)
    inp["w"][:] = 1.0
    qw = tuple(oracle.quantize_e4m3(inp[n]) for n in ("Wg", "Wu", "Wd"))
    Wg, Wu, Wd = (oracle.dequantize_e4m3(*p)[0] for p in qw)
    x = W.bits_to_float(inp["x"], "bf16").astype(np.float64)
    xq = rows_e4m3_torch(x)
    g, u = xq @ Wg, xq @ Wu
    h = g / (1.0 + np.exp(-g)) * u
    # h's codes are decided from h as stored, in bf16 (h -> fp32 -> bf16 is
    # the oracle's rounding for these magnitudes)
    hb = W.bits_to_float(W.bf16_bits(h.astype(np.float32)), "bf16").astype(np.float64)
    if mirror:
        h = hb
    ref = rows_e4m3_torch(hb) @ Wd
    y = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw, act_e4m3=True, mirror=False)
    if not mirror:
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    # the stage view returns h before its quantization and ys after it
    rows = np.arange(T, dtype=np.int64)
    hh, ys = oracle.expert_rows(inp["x"], rows, np.zeros(T, np.int32), np.ones(T, np.float32),
                                *qw, act_e4m3=True, mirror=mirror)
    if mirror:
        assert np.array_equal(hh, h)
    else:
        assert np.allclose(hh, g / (1.0 + np.exp(-g)) * u, rtol=1e-12, atol=1e-15)
    assert np.allclose(ys, ref, rtol=1e-12, atol=1e-15)


def test_gate_up_e4m3_activations_equal_layer_on_dequantized_rows():
    # the gate/up half through the already pinned path: h from E4M3 rows ==
    # h of the rows' dequantized values (exact in bf16)
    T, d, E, k, f = 10, 64, 3, 2, 32
    inp = W.make_layer(T, d, E, k, f, seed=11)
    qw = tuple(oracle.quantize_e4m3(inp[n]) for n in ("Wg", "Wu", "Wd"))
    q, e = oracle.quantize_rows_e4m3(inp["x"])
    deq = np.array([[oracle.e4m3_value(c) for c in row] for row in q]) * (2.0 ** e)[:, None]
    xd = W.bf16_bits(deq.astype(np.float32))
    assert np.array_equal(W.bits_to_float(xd, "bf16").astype(np.float64), deq)
    rows = np.arange(T, dtype=np.int64)
    re = (np.arange(T) % E).astype(np.int32)
    rw = np.ones(T, np.float32)
    h8, _ = oracle.expert_rows(inp["x"], rows, re, rw, *qw, act_e4m3=True)
    hd, _ = oracle.expert_rows(xd, rows, re, rw, *qw)
    assert np.array_equal(h8, hd)
