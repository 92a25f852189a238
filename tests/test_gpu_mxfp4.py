"""MXFP4 expert weights on the GPU vs the oracle.

moe_quantize_mxfp4 must give the oracle's codes and scale exponents bit for
bit.  Every dequantized MXFP4 weight is a bf16 value, so the GEMMs on MXFP4
weights must equal the bf16 GEMMs on the oracle's dequantized weights bit
for bit: that pins the decoding into tensor memory (the 4-bit codes, their
nibble order, the per-block scales and the lane / column layout the MMAs
read them in).

The library stores codes along K ([E, M, K/2] bytes, eight codes to a
little-endian 32-bit word: k = 8i + 2j at bits 4j, k = 8i + 2j + 1 at bits
16 + 4j); the oracle's are [E, K, M/2] (feature m even in the low nibble).
``kmajor`` turns the oracle's into the library's layout (a pure
re-arrangement of the same 4-bit codes).

The whole layer is checked against the oracle's layer on the dequantized
weights (the layer bar) and against the bf16 layer on them (bit for
bit)."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import dev, dev16, host16, host_f, inputs, layer_tolerance, sample_tokens

pytestmark = pytest.mark.gpu


def kmajor(codes):
    """Oracle codes [E, K, M/2] -> the library's [E, M, K/2]: per group of
    eight k, bytes (k0 | k2 << 4, k4 | k6 << 4, k1 | k3 << 4, k5 | k7 << 4)."""
    E, K, M2 = codes.shape
    nib = np.empty((E, K, 2 * M2), dtype=np.uint8)
    nib[:, :, 0::2] = codes & 0x0F
    nib[:, :, 1::2] = codes >> 4
    t = nib.transpose(0, 2, 1).reshape(E, 2 * M2, K // 8, 8)  # [E, M, K/8, 8]
    out = np.empty((E, 2 * M2, K // 8, 4), dtype=np.uint8)
    for b, (lo, hi) in enumerate(((0, 2), (4, 6), (1, 3), (5, 7))):
        out[..., b] = t[..., lo] | (t[..., hi] << 4)
    return np.ascontiguousarray(out.reshape(E, 2 * M2, K // 2))


def gpu_quantize(bits):
    m = B.quantize_mxfp4(dev16(bits))
    torch.cuda.synchronize()
    return m.codes.cpu().numpy(), m.scales.cpu().numpy()


@pytest.mark.parametrize("E,K,M,std", [(3, 64, 64, 0.02), (2, 96, 704, 1.0), (2, 32, 2, 300.0),
                                       (1, 128, 192, 1e-30)])
def test_quantize_matches_oracle_bitwise(E, K, M, std):
    rng = np.random.default_rng(E * K + M)
    Wf = (rng.standard_normal((E, K, M)) * std).astype(np.float32)
    Wf[0, :32, 1 % M] = 0.0                   # a zero block
    Wf[0, 32 % K:, 0] *= 1e-6                 # a block far below its column
    Wf[-1, 5, :] = -0.0                       # negative zeros
    if M >= 4:
        Wf[0, :8, 3] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]  # midpoints at exponent 0
        Wf[0, 8:32, 3] = 0.0
    bits = W.bf16_bits(Wf)
    c, s = gpu_quantize(bits)
    co, so = oracle.quantize_mxfp4(bits)
    assert np.array_equal(s, so)
    assert np.array_equal(c, kmajor(co))


def test_quantize_workload_weights_sampled_experts():
    wl = W.workload(3)
    inp = inputs(3)
    c, s = gpu_quantize(inp["Wd"])
    for e in (0, 77, wl.E - 1):
        co, so = oracle.quantize_mxfp4(inp["Wd"][e:e + 1])
        assert np.array_equal(c[e:e + 1], kmajor(co)) and np.array_equal(s[e:e + 1], so)


def mx_dev(bits):
    """Oracle MXFP4 weights on the device, and their dequantized bf16 weights."""
    codes, scales = oracle.quantize_mxfp4(bits)
    return B.Mxfp4(dev(kmajor(codes)), dev(scales)), dev16(oracle.dequantize_mxfp4(codes, scales))


def staged(inp, E, tm):
    p = oracle.plan(inp["ids"], inp["w"], E, tm)
    xs = oracle.gather(inp["x"], p["srt_tok"])
    return p, xs


def to_cap(a, cap):
    out = np.zeros((cap,) + a.shape[1:], dtype=a.dtype)
    out[:len(a)] = a
    return out


@pytest.mark.parametrize("T,d,E,k,f,tm", [
    (40, 64, 3, 2, 64, 16),       # one K step, M tile half empty
    (100, 192, 5, 3, 192, 16),    # partial feature tiles on both GEMMs (192 = 128 + 64)
    (300, 128, 2, 1, 256, 32),    # experts over 128 rows
    (257, 256, 6, 4, 704, 16),    # f = 5.5 x 128: the last tile half outside the weights
])
def test_gemms_equal_bf16_gemms_on_dequantized_weights(T, d, E, k, f, tm):
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=T + 3 * f, skip_frac=0.1)
    p, xs = staged(inp, E, tm)
    cap = B.capacity(T, k, E, tm)
    offsets = dev(p["offsets"])
    (mg, g16), (mu, u16), (md, d16w) = (mx_dev(inp[n]) for n in ("Wg", "Wu", "Wd"))
    xs_d = dev16(to_cap(xs, cap))
    H4 = B.ffn_gate_up_mxfp4(xs_d, mg, mu, offsets, cap)
    H16 = B.ffn_gate_up(xs_d, g16, u16, offsets, cap)
    R = p["R_pad"]
    assert torch.equal(H4[:R].view(torch.int16), H16[:R].view(torch.int16))
    srt_w = dev(to_cap(p["srt_w"], cap))
    Y4 = B.ffn_down_mxfp4(H16, md, offsets, srt_w, cap)
    Y16 = B.ffn_down(H16, d16w, offsets, srt_w, cap)
    assert torch.equal(Y4[:R].view(torch.int16), Y16[:R].view(torch.int16))
    # and against the oracle's fp64 stage on the dequantized weights
    real = np.nonzero(p["srt_tok"] >= 0)[0]
    row_e = (np.searchsorted(p["offsets"], np.arange(R), side="right") - 1).astype(np.int32)
    host = [oracle.dequantize_mxfp4(*oracle.quantize_mxfp4(inp[n])) for n in ("Wg", "Wu", "Wd")]
    h_ref, _ = oracle.expert_rows(xs, real, row_e[real], p["srt_w"][real], *host)
    ok, err, bound = layer_tolerance(
        W.bits_to_float(host16(H4)[real], "bf16").astype(np.float64), h_ref)
    assert ok, (err, bound)


def test_gemms_large_weights_take_the_fp32_scaling():
    # blocks with |W| >= 8 (S > 128) decode through the f16 conversion and an
    # fp32 multiply; mixed with ordinary blocks in the same tiles
    T, d, E, k, f, tm = 120, 128, 3, 2, 192, 16
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=77, skip_frac=0.0)
    for n in ("Wg", "Wu", "Wd"):
        Wf = W.bits_to_float(inp[n], "bf16").astype(np.float32)
        Wf[:, :, ::3] *= 4000.0      # every third output feature: |W| up to ~300
        inp[n] = W.bf16_bits(Wf)
    p, xs = staged(inp, E, tm)
    cap = B.capacity(T, k, E, tm)
    offsets = dev(p["offsets"])
    (mg, g16), (mu, u16), (md, d16w) = (mx_dev(inp[n]) for n in ("Wg", "Wu", "Wd"))
    assert int(mg.scales.max()) > 128 and int(mg.scales.min()) <= 128
    xs_d = dev16(to_cap(xs, cap))
    R = p["R_pad"]
    H4 = B.ffn_gate_up_mxfp4(xs_d, mg, mu, offsets, cap)
    H16 = B.ffn_gate_up(xs_d, g16, u16, offsets, cap)
    assert torch.equal(H4[:R].view(torch.int16), H16[:R].view(torch.int16))
    srt_w = dev(to_cap(p["srt_w"], cap))
    Y4 = B.ffn_down_mxfp4(H16, md, offsets, srt_w, cap)
    Y16 = B.ffn_down(H16, d16w, offsets, srt_w, cap)
    assert torch.equal(Y4[:R].view(torch.int16), Y16[:R].view(torch.int16))


def layer_case(inp, tm, tokens=None):
    (mg, g16), (mu, u16), (md, d16w) = (mx_dev(inp[n]) for n in ("Wg", "Wu", "Wd"))
    x, ids, w = dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])
    y4 = B.layer_forward_mxfp4(x, ids, w, mg, mu, md, tm)
    y16 = B.layer_forward(x, ids, w, g16, u16, d16w, tm)
    torch.cuda.synchronize()
    assert torch.equal(y4.view(torch.int16), y16.view(torch.int16))
    host = [oracle.dequantize_mxfp4(*oracle.quantize_mxfp4(inp[n])) for n in ("Wg", "Wu", "Wd")]
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *host, tokens=tokens)
    got = host_f(y4) if tokens is None else host_f(y4)[tokens]
    ok, err, bound = layer_tolerance(got, ref)
    assert ok, (err, bound)
    return got


@pytest.mark.parametrize("T,d,E,k,f,tm,skip", [
    (50, 64, 4, 2, 64, 16, 0.0),
    (123, 192, 9, 3, 192, 16, 0.2),
    (200, 128, 70, 4, 704, 16, 0.1),
    (9000, 64, 64, 8, 64, 16, 0.05),     # the multi-kernel plan
])
def test_layer_small_shapes_full_output(T, d, E, k, f, tm, skip):
    layer_case(W.make_layer(T, d, E, k, f, tm=tm, seed=5 * T + E, skip_frac=skip), tm)


def test_layer_full_size_sampled_tokens_and_error_vs_bf16_weights():
    # the full page-1-scale layer on MXFP4 weights: within the bar of the
    # oracle's layer on the dequantized weights; its distance from the layer
    # on the original bf16 weights is the quantization error, reported
    wl = W.workload(3)
    inp = inputs(3)
    toks = sample_tokens(inp["ids"], 24, seed=4)
    got = layer_case(inp, wl.tm, tokens=toks)
    ref16 = oracle.layer(inp["x"], inp["ids"], inp["w"], inp["Wg"], inp["Wu"], inp["Wd"],
                         tokens=toks)
    rel = float(np.linalg.norm(got - ref16) / np.linalg.norm(ref16))
    print(f"MXFP4 layer vs the bf16-weight oracle on {len(toks)} tokens: rel-L2 {rel:.3e}, "
          f"max err {np.max(np.abs(got - ref16)):.3e}")
    assert rel < 0.25  # 4-bit weights: the quantization error, not a bug, dominates


def test_moe_layer_quantized_mxfp4_and_determinism():
    wl = W.workload(1)
    inp = inputs(1)
    Wg, Wu, Wd = (dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    layer = B.MoeLayer.quantized_mxfp4(Wg, Wu, Wd, tm=wl.tm)
    x, ids, w = dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])
    a = layer.forward(x, ids, w)
    b = layer.forward(x, ids, w)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert B.read_status(layer._ws) == 0
    host = [oracle.dequantize_mxfp4(*oracle.quantize_mxfp4(inp[n])) for n in ("Wg", "Wu", "Wd")]
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *host)
    ok, err, bound = layer_tolerance(host_f(a), ref)
    assert ok, (err, bound)
