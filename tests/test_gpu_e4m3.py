"""E4M3 expert weights on the GPU vs the oracle.

moe_quantize_e4m3 must give the oracle's codes and scales bit for bit.  The
E4M3 GEMMs are checked stage by stage against the oracle with the same
codes and scales (the layer bar, max|gpu - ref| <= 1e-2 * max|ref| + 1e-3),
and bit for bit against the bf16 GEMMs on weights whose dequantized values
are exact in bf16 (power-of-two scales): that pins the in-shared-memory
widening and its swizzled layout.  The whole layer, its host entry point and
its determinism are checked as for bf16."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import dev, dev16, host16, host_f, inputs, layer_tolerance, sample_tokens

pytestmark = pytest.mark.gpu


def q_dev(qs):
    q, s = qs
    return dev(q), dev(s)


def gpu_quantize(bits):
    q, s = B.quantize_e4m3(dev16(bits))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("E,K,M,scale", [(3, 64, 64, 0.02), (5, 200, 320, 1.0), (2, 96, 704, 3e-3)])
def test_quantize_matches_oracle_bitwise(E, K, M, scale):
    rng = np.random.default_rng(E * K + M)
    Wf = (rng.standard_normal((E, K, M)) * scale).astype(np.float32)
    Wf[0, :, 3] = 0.0                                          # zero column: scale 1
    Wf[1 % E, :, 5] *= 1e-30                                   # tiny column
    Wf[:, 7, :] = -1e-12                                       # rounds to -0 in most columns
    bits = W.bf16_bits(Wf)
    q, s = gpu_quantize(bits)
    qo, so = oracle.quantize_e4m3(bits)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))
    assert np.array_equal(q, qo)


def test_quantize_workload_weights_sampled_experts():
    wl = W.workload(3)
    inp = inputs(3)
    q, s = gpu_quantize(inp["Wg"])
    for e in (0, 77, wl.E - 1):
        qo, so = oracle.quantize_e4m3(inp["Wg"][e:e + 1])
        assert np.array_equal(q[e:e + 1], qo) and np.array_equal(s[e:e + 1], so)


def staged(inp, E, tm):
    p = oracle.plan(inp["ids"], inp["w"], E, tm)
    xs = oracle.gather(inp["x"], p["srt_tok"])
    real = np.nonzero(p["srt_tok"] >= 0)[0]
    row_e = (np.searchsorted(p["offsets"], np.arange(p["R_pad"]), side="right") - 1).astype(np.int32)
    return p, xs, real, row_e


def to_cap(a, cap, fill=0):
    out = np.full((cap,) + a.shape[1:], fill, dtype=a.dtype)
    out[:len(a)] = a
    return out


def run_stages(inp, E, d, f, tm, qw, nsample=None, seed=0):
    """gate/up and down with E4M3 weights qw = ((qg, sg), (qu, su), (qd, sd))
    (host arrays) against the oracle on the real rows (or a sample)."""
    p, xs, real, row_e = staged(inp, E, tm)
    T, k = inp["ids"].shape
    cap = B.capacity(T, k, E, tm)
    offsets = dev(p["offsets"])
    dq = [q_dev(w) for w in qw]
    H = B.ffn_gate_up_e4m3(dev16(to_cap(xs, cap)), dq[0], dq[1], offsets, cap)
    rows = real
    if nsample is not None and len(real) > nsample:
        rows = np.unique(np.random.default_rng(seed).choice(real, nsample, replace=False))
    h_ref, _ = oracle.expert_rows(xs, rows, row_e[rows], p["srt_w"][rows], *qw)
    Hh = host16(H)
    ok, err, bound = layer_tolerance(W.bits_to_float(Hh[rows], "bf16").astype(np.float64), h_ref)
    assert ok, f"gate/up e4m3: max err {err} > {bound}"
    pad = np.nonzero(p["srt_tok"] < 0)[0]
    assert np.all(Hh[pad] == 0)
    hm, ysm = oracle.expert_rows(xs, rows, row_e[rows], p["srt_w"][rows], *qw, mirror=True)
    Hin = np.zeros((cap, f), np.uint16)
    Hin[rows] = W.bf16_bits(hm.astype(np.float32))
    Ys = host16(B.ffn_down_e4m3(dev16(Hin), dq[2], offsets, dev(to_cap(p["srt_w"], cap)), cap))
    ok, err, bound = layer_tolerance(W.bits_to_float(Ys[rows], "bf16").astype(np.float64), ysm)
    assert ok, f"down e4m3: max err {err} > {bound}"
    return H, Ys


def quantized(inp):
    return tuple(oracle.quantize_e4m3(inp[n]) for n in ("Wg", "Wu", "Wd"))


@pytest.mark.parametrize("T,d,E,k,f,tm", [
    (40, 64, 3, 2, 64, 16),      # one K step; the E4M3 box of 128 features is half outside M
    (100, 192, 5, 3, 192, 16),   # down's second 128-feature tile is half outside d
    (300, 128, 2, 1, 256, 32),   # experts with several chunks
    (257, 256, 6, 4, 704, 16),   # f = 5.5 x 128
    (64, 320, 40, 2, 128, 16),   # many small experts
])
def test_e4m3_stages_all_rows(T, d, E, k, f, tm):
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=T + f + 1)
    run_stages(inp, E, d, f, tm, quantized(inp))


def pow2_quantized(E, K, M, seed):
    """Random codes with power-of-two scales, and the bf16 weights equal to
    their dequantized values (exact)."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(E, K, M)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x30                               # no NaN codes
    s = (2.0 ** rng.integers(-8, -5, size=(E, M))).astype(np.float32)
    bits = W.bf16_bits(oracle.dequantize_e4m3(q, s).astype(np.float32))
    return (q, s), bits


@pytest.mark.parametrize("T,d,E,k,f", [(150, 192, 4, 2, 320), (90, 128, 3, 3, 704)])
def test_e4m3_gemms_bit_equal_to_bf16_on_exact_weights(T, d, E, k, f):
    inp = W.make_layer(T, d, E, k, f, seed=9, weights=False)
    g8, gb = pow2_quantized(E, d, f, 1)
    u8, ub = pow2_quantized(E, d, f, 2)
    d8, db = pow2_quantized(E, f, d, 3)
    p, xs, real, row_e = staged(inp, E, 16)
    cap = B.capacity(T, k, E, 16)
    offsets = dev(p["offsets"])
    xs_d = dev16(to_cap(xs, cap))
    H8 = B.ffn_gate_up_e4m3(xs_d, q_dev(g8), q_dev(u8), offsets, cap)
    Hb = B.ffn_gate_up(xs_d, dev16(gb), dev16(ub), offsets, cap)
    R = p["R_pad"]
    assert torch.equal(H8[:R].view(torch.int16), Hb[:R].view(torch.int16))
    srt_w = dev(to_cap(p["srt_w"], cap))
    Y8 = B.ffn_down_e4m3(Hb, q_dev(d8), offsets, srt_w, cap)
    Yb = B.ffn_down(Hb, dev16(db), offsets, srt_w, cap)
    assert torch.equal(Y8[:R].view(torch.int16), Yb[:R].view(torch.int16))


@pytest.mark.parametrize("cfg", [3, 5])
def test_e4m3_stages_workloads_sampled_rows(cfg):
    wl = W.workload(cfg)
    inp = inputs(cfg)
    # quantize on the GPU (bit-equal to the oracle's, checked above) and
    # hand the codes to the oracle
    qw = []
    for n in ("Wg", "Wu", "Wd"):
        q, s = B.quantize_e4m3(dev16(inp[n]))
        qw.append((q.cpu().numpy(), s.cpu().numpy()))
    run_stages(inp, wl.E, wl.d, wl.f, wl.tm, tuple(qw), nsample=40, seed=cfg)


def test_e4m3_layer_tiny_full_output():
    wl = W.workload(1)
    inp = inputs(1)
    qw = quantized(inp)
    layer = B.MoeLayer(*[q_dev(w) for w in qw], tm=wl.tm)
    y = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
    torch.cuda.synchronize()
    assert B.read_status(layer._ws) == 0
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw)
    ok, err, bound = layer_tolerance(host_f(y), ref)
    assert ok, (err, bound)


@pytest.mark.parametrize("cfg", [3, 5])
def test_e4m3_layer_workloads_sampled_tokens(cfg):
    wl = W.workload(cfg)
    inp = inputs(cfg)
    Wb = [dev16(inp[n]) for n in ("Wg", "Wu", "Wd")]
    layer = B.MoeLayer.quantized(*Wb, tm=wl.tm)
    del Wb
    y = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
    torch.cuda.synchronize()
    assert B.read_status(layer._ws) == 0
    qw = tuple((q.cpu().numpy(), s.cpu().numpy()) for q, s in (layer.Wg, layer.Wu, layer.Wd))
    toks = sample_tokens(inp["ids"], 24, seed=cfg)
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw, tokens=toks)
    ok, err, bound = layer_tolerance(host_f(y)[toks], ref)
    assert ok, (err, bound)
    # determinism: a second run gives the same bits
    y2 = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_e4m3_layer_host_chunks():
    T, d, E, k, f, tm = 200, 256, 8, 4, 192, 16
    chunks = [W.make_layer(T, d, E, k, f, tm=tm, seed=60 + c) for c in range(3)]
    qw = quantized(chunks[0])
    layer = B.MoeLayer(*[q_dev(w) for w in qw], tm=tm)
    xs = [torch.from_numpy(c["x"].view(np.int16)).view(torch.bfloat16).pin_memory() for c in chunks]
    ids = [torch.from_numpy(c["ids"]).pin_memory() for c in chunks]
    ws = [torch.from_numpy(c["w"]).pin_memory() for c in chunks]
    ys = [torch.empty((T, d), dtype=torch.bfloat16).pin_memory() for _ in chunks]
    layer.forward_host_chunks(xs, ids, ws, ys)
    torch.cuda.synchronize()
    for c, inp in enumerate(chunks):
        ref_dev = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])).cpu()
        assert torch.equal(ys[c].view(torch.int16), ref_dev.view(torch.int16))
        ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw)
        ok, err, bound = layer_tolerance(host_f(ys[c]), ref)
        assert ok, (c, err, bound)


# ---- E4M3 activations: gate/up on 8-bit operands (tcgen05 kind::f8f6f4) ----

def kmajor(qs):
    q, s = qs
    return np.ascontiguousarray(q.transpose(0, 2, 1)), s


def test_quantize_kmajor_matches_oracle_transposed():
    rng = np.random.default_rng(3)
    Wf = (rng.standard_normal((3, 192, 320)) * 0.05).astype(np.float32)
    bits = W.bf16_bits(Wf)
    q, s = B.quantize_e4m3(dev16(bits), kmajor=True)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_e4m3(bits)
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(q.cpu().numpy(), kmajor((qo, so))[0])


def test_gather_e4m3_matches_oracle_rows():
    T, d, E, k = 300, 256, 7, 3
    inp = W.make_layer(T, d, E, k, 64, seed=21, skip_frac=0.1, weights=False)
    xf = W.bits_to_float(inp["x"], "bf16").astype(np.float32)
    xf[5] *= 1e6                                               # exponents far from 0
    xf[9] *= 1e-6
    xf[11] = 0.0                                               # zero row: e = 0
    xf[13, :] = 448.0                                          # exactly at the top code
    x = W.bf16_bits(xf)
    p = oracle.plan(inp["ids"], inp["w"], E, 16)
    cap = B.capacity(T, k, E, 16)
    xs8, xexp = B.gather_e4m3(dev16(x), dev(to_cap(p["srt_tok"], cap, fill=-1)),
                              dev(p["offsets"]), E, cap)
    torch.cuda.synchronize()
    R = p["R_pad"]
    q = xs8.cpu().numpy()[:R]
    e = xexp.cpu().numpy()[:R]
    xs = oracle.gather(x, p["srt_tok"])
    qo, eo = oracle.quantize_rows_e4m3(xs)
    assert np.array_equal(e, eo)
    assert np.array_equal(q, qo)
    pad = p["srt_tok"] < 0
    assert np.all(q[pad] == 0) and np.all(e[pad] == 0)


def run_f8_gate_up(inp, E, d, f, tm, qw, nsample=None, seed=0):
    p, xs, real, row_e = staged(inp, E, tm)
    T, k = inp["ids"].shape
    cap = B.capacity(T, k, E, tm)
    offsets = dev(p["offsets"])
    x8, xe = B.gather_e4m3(dev16(inp["x"]), dev(to_cap(p["srt_tok"], cap, fill=-1)), offsets, E,
                           cap)
    H = B.ffn_gate_up_f8(x8, xe, q_dev(kmajor(qw[0])), q_dev(kmajor(qw[1])), offsets, cap)
    rows = real
    if nsample is not None and len(real) > nsample:
        rows = np.unique(np.random.default_rng(seed).choice(real, nsample, replace=False))
    h_ref, _ = oracle.expert_rows(xs, rows, row_e[rows], p["srt_w"][rows], *qw, act_e4m3=True)
    Hh = host16(H)
    ok, err, bound = layer_tolerance(W.bits_to_float(Hh[rows], "bf16").astype(np.float64), h_ref)
    assert ok, f"gate/up f8: max err {err} > {bound}"
    assert np.all(Hh[np.nonzero(p["srt_tok"] < 0)[0]] == 0)


@pytest.mark.parametrize("T,d,E,k,f,tm", [
    (40, 128, 3, 2, 64, 16),     # one K stage; half the 128-feature box outside f
    (257, 256, 6, 4, 704, 16),   # f = 5.5 x 128
    (300, 384, 2, 1, 256, 32),   # experts with several chunks
    (64, 128, 40, 2, 128, 16),   # many small experts
])
def test_f8_gate_up_all_rows(T, d, E, k, f, tm):
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=T + d)
    run_f8_gate_up(inp, E, d, f, tm, quantized(inp))


@pytest.mark.parametrize("cfg", [3, 5])
def test_f8_gate_up_workloads_sampled_rows(cfg):
    wl = W.workload(cfg)
    inp = inputs(cfg)
    qw = []
    for n in ("Wg", "Wu", "Wd"):
        q, s = B.quantize_e4m3(dev16(inp[n]))
        qw.append((q.cpu().numpy(), s.cpu().numpy()))
    run_f8_gate_up(inp, wl.E, wl.d, wl.f, wl.tm, tuple(qw), nsample=40, seed=cfg)


def test_rows_e4m3_matches_oracle():
    rng = np.random.default_rng(31)
    cap, f = 200, 192
    Hf = (rng.standard_normal((cap, f)) * 3.0).astype(np.float32)
    Hf[7] *= 1e-9
    Hf[8] = 0.0
    H = W.bf16_bits(Hf)
    R = 160                                                    # rows past offsets[E] untouched
    offsets = np.array([0, 64, 64, 160], np.int32)
    H8 = torch.full((cap, f), 0x55, dtype=torch.uint8, device="cuda")
    hexp = torch.full((cap,), 99, dtype=torch.int32, device="cuda")
    B.rows_e4m3(dev16(H), dev(offsets), 3, cap, H8, hexp)
    torch.cuda.synchronize()
    qo, eo = oracle.quantize_rows_e4m3(H[:R])
    assert np.array_equal(H8.cpu().numpy()[:R], qo) and np.array_equal(hexp.cpu().numpy()[:R], eo)
    assert np.all(H8.cpu().numpy()[R:] == 0x55) and np.all(hexp.cpu().numpy()[R:] == 99)


@pytest.mark.parametrize("T,d,E,k,f,tm", [
    (40, 128, 3, 2, 64, 16),     # one K stage, half of it past f (zero-filled)
    (100, 192, 5, 3, 704, 16),   # d = 1.5 x 128: down's second feature tile half outside
    (300, 256, 2, 1, 384, 32),   # experts with several chunks
])
def test_f8_down_all_rows(T, d, E, k, f, tm):
    # down on E4M3 H rows: the oracle's mirror h (bf16) quantized per row by
    # the oracle feeds the GPU, against the oracle's E4M3-activation mirror
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=T + f + 7)
    qw = quantized(inp)
    p, xs, real, row_e = staged(inp, E, tm)
    cap = B.capacity(T, k, E, tm)
    hm, ysm = oracle.expert_rows(xs, real, row_e[real], p["srt_w"][real], *qw, mirror=True,
                                 act_e4m3=True)
    Hin = np.zeros((cap, f), np.uint16)
    Hin[real] = W.bf16_bits(hm.astype(np.float32))
    q8, e8 = oracle.quantize_rows_e4m3(Hin)
    Ys = host16(B.ffn_down_f8(dev(q8), dev(e8), q_dev(kmajor(qw[2])), dev(p["offsets"]),
                              dev(to_cap(p["srt_w"], cap)), cap))
    ok, err, bound = layer_tolerance(W.bits_to_float(Ys[real], "bf16").astype(np.float64), ysm)
    assert ok, f"down f8: max err {err} > {bound}"
    assert np.all(Ys[np.nonzero(p["srt_tok"] < 0)[0]] == 0)


def test_f8_layer_tiny_full_output():
    wl = W.workload(1)
    inp = inputs(1)
    qw = quantized(inp)
    layer = B.MoeLayer(*[q_dev(kmajor(w)) for w in qw], tm=wl.tm, act_e4m3=True)
    y = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
    torch.cuda.synchronize()
    assert B.read_status(layer._ws) == 0
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw, act_e4m3=True)
    ok, err, bound = layer_tolerance(host_f(y), ref)
    assert ok, (err, bound)


@pytest.mark.parametrize("cfg", [3, 5])
def test_f8_layer_workloads_sampled_tokens(cfg):
    wl = W.workload(cfg)
    inp = inputs(cfg)
    Wb = [dev16(inp[n]) for n in ("Wg", "Wu", "Wd")]
    layer = B.MoeLayer.quantized(*Wb, tm=wl.tm, act_e4m3=True)
    del Wb
    y = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
    torch.cuda.synchronize()
    assert B.read_status(layer._ws) == 0
    # the oracle takes the gate/up codes in the weights' own layout
    tr = lambda qs: (np.ascontiguousarray(qs[0].cpu().numpy().transpose(0, 2, 1)),
                     qs[1].cpu().numpy())
    qw = (tr(layer.Wg), tr(layer.Wu), tr(layer.Wd))
    toks = sample_tokens(inp["ids"], 24, seed=cfg)
    ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw, tokens=toks, act_e4m3=True)
    ok, err, bound = layer_tolerance(host_f(y)[toks], ref)
    assert ok, (err, bound)
    y2 = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"]))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_f8_layer_host_chunks():
    T, d, E, k, f, tm = 200, 256, 8, 4, 192, 16
    chunks = [W.make_layer(T, d, E, k, f, tm=tm, seed=80 + c) for c in range(3)]
    qw = quantized(chunks[0])
    layer = B.MoeLayer(*[q_dev(kmajor(w)) for w in qw], tm=tm, act_e4m3=True)
    xs = [torch.from_numpy(c["x"].view(np.int16)).view(torch.bfloat16).pin_memory() for c in chunks]
    ids = [torch.from_numpy(c["ids"]).pin_memory() for c in chunks]
    ws = [torch.from_numpy(c["w"]).pin_memory() for c in chunks]
    ys = [torch.empty((T, d), dtype=torch.bfloat16).pin_memory() for _ in chunks]
    layer.forward_host_chunks(xs, ids, ws, ys)
    torch.cuda.synchronize()
    for c, inp in enumerate(chunks):
        ref_dev = layer.forward(dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])).cpu()
        assert torch.equal(ys[c].view(torch.int16), ref_dev.view(torch.int16))
        ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw, act_e4m3=True)
        ok, err, bound = layer_tolerance(host_f(ys[c]), ref)
        assert ok, (c, err, bound)


@pytest.mark.parametrize("T,d,E,k,f,tm,skip", [
    (300, 128, 4096, 4, 64, 16, 0.0),    # E at its limit: the largest chunk table
    (9000, 128, 64, 8, 128, 16, 0.05),   # T*k above 16 x 4096: the multi-kernel plan
    (123, 192, 9, 3, 192, 16, 0.2),      # ragged tiles, skipped slots, d = 1.5 x 128
])
def test_f8_and_e4m3_layers_at_the_limits(T, d, E, k, f, tm, skip):
    inp = W.make_layer(T, d, E, k, f, tm=tm, seed=5 * T + E, skip_frac=skip)
    qw = quantized(inp)
    x, ids, w = dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])
    for act in (False, True):
        weights = [q_dev(kmajor(q)) if act else q_dev(q) for q in qw]
        layer = B.MoeLayer(*weights, tm=tm, act_e4m3=act)
        y = layer.forward(x, ids, w)
        torch.cuda.synchronize()
        assert B.read_status(layer._ws) == 0
        ref = oracle.layer(inp["x"], inp["ids"], inp["w"], *qw, act_e4m3=act)
        ok, err, bound = layer_tolerance(host_f(y), ref)
        assert ok, (act, err, bound)


@pytest.mark.parametrize("cfg", [1, 3])
def test_f8_layer_equals_its_stages_bitwise(cfg):
    # the layer quantizes each token once and gathers its codes; the stage
    # calls quantize each routed row: the same codes, so the same bits
    wl = W.workload(cfg)
    inp = inputs(cfg)
    layer = B.MoeLayer.quantized(*[dev16(inp[n]) for n in ("Wg", "Wu", "Wd")], tm=wl.tm,
                                 act_e4m3=True)
    x, ids, w = dev16(inp["x"]), dev(inp["ids"]), dev(inp["w"])
    y = layer.forward(x, ids, w)
    cap = B.capacity(wl.T, wl.k, wl.E, wl.tm)
    o = B.plan(ids, w, wl.E, wl.tm, cap=cap)
    x8, xe = B.gather_e4m3(x, o["srt_tok"], o["offsets"], wl.E, cap)
    H = B.ffn_gate_up_f8(x8, xe, layer.Wg, layer.Wu, o["offsets"], cap)
    H8, he = B.rows_e4m3(H, o["offsets"], wl.E, cap)
    Ys = B.ffn_down_f8(H8, he, layer.Wd, o["offsets"], o["srt_w"], cap)
    y2 = B.combine(Ys, o["pos"])
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
