"""Pins of the oracle's MXFP4 weights (CPU).

MXFP4 is the 4-bit format of the OCP Microscaling (MX) specification: E2M1
elements (1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; the
magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, no infinities or NaN) in blocks of
32 along the reduction axis, each block sharing a power-of-two scale whose
exponent is stored as an unsigned byte (value 2^(S-127)).  The block's
exponent is floor(log2(max |v|)) minus the exponent of E2M1's largest
normal (2), and each element is the nearest E2M1 value to v / scale, ties to
the even code, past 6 saturated.

The pins below check the oracle against that definition by other means: the
value set the format lists, a brute-force nearest search over all 16 codes,
hand-built blocks on the grid, at midpoints, saturating, zero and at the
ends of the exponent range, the error bound of the rounding, and round trips.
"""
import numpy as np
import pytest

import oracle
from moe_prefill_routing_gb300 import workload as W

# the format's value set, codes 0..7 (codes 8..15 are their negatives)
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bits(values):
    return W.bf16_bits(np.asarray(values, np.float32))


def unpack(codes):
    """[E, K, M/2] bytes -> [E, K, M] 4-bit codes (feature m even = low nibble)."""
    out = np.empty(codes.shape[:-1] + (2 * codes.shape[-1],), np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def brute_force(Wf):
    """Independent reference: per (expert, block, feature) the exponent from
    frexp of the block's max magnitude, then each element the nearest of the
    16 code values times 2^x, ties to the code with mantissa bit 0, the sign
    of a zero result taken from the input."""
    E, K, M = Wf.shape
    table = np.array(E2M1_MAGNITUDES + [-v for v in E2M1_MAGNITUDES])
    codes = np.zeros((E, K, M), np.uint8)
    scales = np.zeros((E, K // 32, M), np.uint8)
    for e in range(E):
        for b in range(K // 32):
            for m in range(M):
                blk = Wf[e, 32 * b:32 * b + 32, m].astype(np.float64)
                amax = np.max(np.abs(blk))
                if amax == 0:
                    x = -127
                else:
                    x = int(np.frexp(amax)[1]) - 1 - 2
                    x = max(-127, min(127, x))
                scales[e, b, m] = x + 127
                for i, v in enumerate(blk):
                    cand = table * 2.0 ** x
                    if abs(v) >= 6 * 2.0 ** x:
                        c = 7
                    else:
                        dist = np.abs(cand[:8] - abs(v))
                        best = np.flatnonzero(dist == dist.min())
                        c = int(best[0]) if len(best) == 1 else int([q for q in best if q % 2 == 0][0])
                    if np.signbit(v):
                        c |= 8
                    codes[e, 32 * b + i, m] = c
    return codes, scales


def test_e2m1_values_are_the_formats_value_set():
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert vals[:8] == E2M1_MAGNITUDES
    assert vals[8:] == [-v for v in E2M1_MAGNITUDES]
    assert np.signbit(vals[8]) and not np.signbit(vals[0])


@pytest.mark.parametrize("std,seed", [(0.02, 0), (1.0, 1), (300.0, 2), (1e-30, 3)])
def test_quantize_matches_brute_force(std, seed):
    rng = np.random.default_rng(seed)
    E, K, M = 2, 64, 6
    Wf = (rng.standard_normal((E, K, M)) * std).astype(np.float32)
    Wf[0, :32, 0] = 0.0                     # a zero block
    Wf[1, 32:, 3] *= 1e-3                   # a block far smaller than its neighbours
    Wb = bits(Wf)
    codes, scales = oracle.quantize_mxfp4(Wb)
    ref_c, ref_s = brute_force(W.bits_to_float(Wb, "bf16"))
    assert np.array_equal(scales, ref_s)
    assert np.array_equal(unpack(codes), ref_c)


def test_blocks_on_the_grid_round_trip_exactly():
    # every E2M1 magnitude times 2^-5 with the block maximum 6 * 2^-5, so
    # the block exponent is -5 and every element is representable
    mags = np.array(E2M1_MAGNITUDES * 4, np.float32)[:32] * 2.0 ** -5
    mags[0] = 6 * 2.0 ** -5
    signs = np.where(np.arange(32) % 3 == 0, -1.0, 1.0).astype(np.float32)
    Wf = (mags * signs).reshape(1, 32, 1).repeat(2, axis=2)
    Wb = bits(Wf)
    codes, scales = oracle.quantize_mxfp4(Wb)
    assert np.all(scales == 127 - 5)
    assert np.array_equal(oracle.dequantize_mxfp4(codes, scales), Wb)


def test_midpoints_round_to_the_even_code():
    # the seven midpoints between neighbouring magnitudes (block exponent 0:
    # the first element is 6, so max = 6 and x = floor(log2 6) - 2 = 0)
    mid = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    expect = [7, 0, 2, 2, 4, 4, 6, 6]  # codes: 6 | 0 | 1.0 | 1.0 | 2 | 2 | 4 | 4
    Wf = np.zeros((1, 32, 2), np.float32)
    Wf[0, :8, 0] = mid
    Wf[0, :8, 1] = [-v for v in mid]
    codes, scales = oracle.quantize_mxfp4(bits(Wf))
    c = unpack(codes)
    assert scales[0, 0, 0] == 127 and scales[0, 0, 1] == 127
    assert c[0, :8, 0].tolist() == expect
    assert c[0, :8, 1].tolist() == [v | 8 for v in expect]


def test_saturation_zero_and_exponent_range():
    Wf = np.zeros((1, 32, 6), np.float32)
    Wf[0, 0, 0] = 7.5          # max 7.5: x = 0 and 7.5 -> 6 (saturated), 5.0 a tie -> 4
    Wf[0, 1, 0] = 5.0
    Wf[0, :, 1] = -0.0         # negative zeros: codes 8, scale byte 0
    Wf[0, 0, 2] = 2.0 ** -133  # bf16 subnormals: exponent clamped to -127
    Wf[0, 1, 2] = 2.0 ** -131
    Wf[0, 0, 3] = 2.0 ** 127   # the top: x = 125, scale byte 252
    Wf[0, 1, 3] = -3.0 * 2.0 ** 125
    codes, scales = oracle.quantize_mxfp4(bits(Wf))
    c = unpack(codes)
    assert scales[0, 0, 0] == 127 and c[0, 0, 0] == 7 and c[0, 1, 0] == 6
    assert scales[0, 0, 1] == 0 and np.all(c[0, :, 1] == 8)
    assert scales[0, 0, 2] == 0
    # 2^-133 / 2^-127 = 2^-6 rounds to 0; 2^-131 / 2^-127 = 2^-4 also to 0
    assert c[0, 0, 2] == 0 and c[0, 1, 2] == 0
    assert scales[0, 0, 3] == 252 and c[0, 0, 3] == 6 and c[0, 1, 3] == (5 | 8)
    deq = W.bits_to_float(oracle.dequantize_mxfp4(codes, scales), "bf16")
    assert deq[0, 0, 3] == 2.0 ** 127 and deq[0, 1, 3] == -3.0 * 2.0 ** 125


def test_rounding_error_bound_and_idempotence():
    rng = np.random.default_rng(7)
    Wf = (rng.standard_normal((3, 96, 8)) * np.exp(rng.uniform(-8, 8, (3, 1, 8)))).astype(np.float32)
    Wb = bits(Wf)
    codes, scales = oracle.quantize_mxfp4(Wb)
    deq = oracle.dequantize_mxfp4(codes, scales)
    a = W.bits_to_float(Wb, "bf16").astype(np.float64)
    b = W.bits_to_float(deq, "bf16").astype(np.float64)
    x = scales.astype(np.int64) - 127                       # [E, K/32, M]
    X = np.repeat(2.0 ** x, 32, axis=1)                    # per element
    r = np.abs(a) / X                                      # in [0, 8)
    assert np.all(r < 8)
    # half the grid step at |v| / X: 0.25 below 2, 0.5 in [2, 4), 1 in [4, 6);
    # saturation above 6 costs at most 2
    half = np.where(r < 2, 0.25, np.where(r < 4, 0.5, np.where(r < 6, 1.0, 2.0)))
    assert np.all(np.abs(a - b) <= half * X)
    # each block's largest element lands at 4 or more (the exponent is not too large)
    blockmax = np.abs(a).reshape(3, 3, 32, 8).max(axis=2)
    assert np.all(blockmax / 2.0 ** x >= 4)
    # quantizing the dequantized weights gives the same codes and scales
    c2, s2 = oracle.quantize_mxfp4(deq)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)


def test_codes_pack_features_in_nibbles():
    # feature 0 = 1.0 (code 2), feature 1 = -4.0 (code 14), in one byte 0xE2
    Wf = np.zeros((1, 32, 2), np.float32)
    Wf[0, 0, 0], Wf[0, 0, 1] = 1.0, -4.0
    Wf[0, 1, 0], Wf[0, 1, 1] = 4.0, 4.0   # both blocks' max 4: exponent 0
    codes, scales = oracle.quantize_mxfp4(bits(Wf))
    assert codes[0, 0, 0] == 0xE2 and codes[0, 1, 0] == 0x66
    assert scales[0, 0, 0] == scales[0, 0, 1] == 127


def test_mxfp4_layer_is_the_bf16_layer_on_grid_weights():
    # weights already on the MXFP4 grid: dequantize(quantize(W)) == W, so the
    # layer on MXFP4 weights equals the bf16 layer bit for bit
    rng = np.random.default_rng(3)
    E, d, f, T, k = 3, 64, 64, 5, 2
    def grid(shape):
        c = rng.integers(0, 16, size=shape)
        v = np.array([oracle.e2m1_value(int(q)) for q in c.ravel()]).reshape(shape)
        return bits((v * 2.0 ** -6).astype(np.float32))
    Wg, Wu, Wd = grid((E, d, f)), grid((E, d, f)), grid((E, f, d))
    x = bits(rng.standard_normal((T, d)).astype(np.float32))
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, -1], [2, 1]], np.int32)
    w = rng.random((T, k)).astype(np.float32)
    q = [oracle.dequantize_mxfp4(*oracle.quantize_mxfp4(t)) for t in (Wg, Wu, Wd)]
    for a, b in zip(q, (Wg, Wu, Wd)):
        assert np.array_equal(a, b)
    assert np.array_equal(oracle.layer(x, ids, w, *q), oracle.layer(x, ids, w, Wg, Wu, Wd))
