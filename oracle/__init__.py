"""CPU oracle of the routed MoE prefill layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports, links or runs anything here, and this package
imports nothing from the product: the two share only the seeded input
generator, which holds none of the layer's arithmetic.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, -ffp-contract=off);
this module loads it with ctypes, building it with gcc on first use.  Each
function cites the passage it follows in the C source:

* ``plan``        -- the routing plan as a stable counting sort ("Round 4 Track
  C: Prefill MoE Plan ...", section 1 items 1-2 and section 3);
* ``gather``      -- the row gather (same page, section 1 item 4);
* ``layer``       -- the flat (token, expert, weight) job pass and the slot-
  ordered combine ("Batched resident MoE experts on Apple Silicon ...",
  sections 1 and 3);
* ``expert_rows`` / ``combine`` -- the same arithmetic cut at the stage
  boundaries, to check one GPU stage at a time;
* ``quantize_e4m3`` -- expert weights as E4M3 codes with one fp32 scale per
  (expert, output feature) ("Round 4 Track C ...", section 2 runs the
  experts from quantized packs; E4M3 is the OCP 8-bit floating point
  format).  ``layer`` and ``expert_rows`` take such weights as
  ``(codes, scales)`` pairs in place of bf16 arrays;
* ``quantize_mxfp4`` / ``dequantize_mxfp4`` -- expert weights as 4-bit
  MXFP4 (the OCP Microscaling format: E2M1 codes in blocks of 32 along the
  reduction axis with a power-of-two scale each); the dequantized weights
  are exact bf16 values, so the layer on MXFP4 weights is ``layer`` on
  them.

Pins (CPU tests): brute force on tiny inputs, closed forms, a dense numpy
cross-check for a single expert, invariants, and hand-worked fixtures under
``tests/golden/``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
             "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so (gcc, host only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MOE_ORACLE_LIB points the tests' planted-mistake runs at a
            # deliberately broken build of this same source
            path = os.environ.get("MOE_ORACLE_LIB") or build()
            lib = C.CDLL(path)
            P = C.c_void_p
            lib.oracle_plan.restype = C.c_long
            lib.oracle_plan.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_int,
                                        P, P, P, P, P, P, C.c_long]
            lib.oracle_gather.restype = None
            lib.oracle_gather.argtypes = [P, C.c_int, C.c_int, P, C.c_long, P]
            lib.oracle_layer_tokens.restype = C.c_int
            lib.oracle_layer_tokens.argtypes = [P, C.c_int, P, P, P, P, P, C.c_int,
                                                C.c_int, C.c_int, C.c_int, C.c_int,
                                                P, C.c_int, C.c_int, C.c_int, P]
            lib.oracle_expert_rows.restype = C.c_int
            lib.oracle_expert_rows.argtypes = [P, C.c_int, C.c_int, C.c_int, P, C.c_int,
                                               P, P, C.c_int, P, P, P, C.c_int, C.c_int,
                                               P, P]
            lib.oracle_combine.restype = None
            lib.oracle_combine.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P]
            lib.oracle_round_bf16.restype = C.c_double
            lib.oracle_round_bf16.argtypes = [C.c_double]
            lib.oracle_value16.restype = C.c_double
            lib.oracle_value16.argtypes = [C.c_uint16, C.c_int]
            lib.oracle_e4m3_value.restype = C.c_double
            lib.oracle_e4m3_value.argtypes = [C.c_uint8]
            lib.oracle_e4m3_encode.restype = C.c_uint8
            lib.oracle_e4m3_encode.argtypes = [C.c_float]
            lib.oracle_quantize_e4m3.restype = None
            lib.oracle_quantize_e4m3.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
            lib.oracle_e2m1_value.restype = C.c_double
            lib.oracle_e2m1_value.argtypes = [C.c_uint8]
            lib.oracle_quantize_mxfp4.restype = None
            lib.oracle_quantize_mxfp4.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
            lib.oracle_dequantize_mxfp4.restype = C.c_int
            lib.oracle_dequantize_mxfp4.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P]
            lib.oracle_layer_tokens_e4m3.restype = C.c_int
            lib.oracle_layer_tokens_e4m3.argtypes = [P, C.c_int, P, P, P, P, P, P, P, P,
                                                     C.c_int, C.c_int, C.c_int, C.c_int,
                                                     C.c_int, P, C.c_int, C.c_int, C.c_int,
                                                     C.c_int, P]
            lib.oracle_expert_rows_e4m3.restype = C.c_int
            lib.oracle_expert_rows_e4m3.argtypes = [P, C.c_int, C.c_int, C.c_int, P, C.c_int,
                                                    P, P, C.c_int, P, P, P, P, P, P, C.c_int,
                                                    C.c_int, C.c_int, P, P]
            lib.oracle_quantize_rows_e4m3.restype = None
            lib.oracle_quantize_rows_e4m3.argtypes = [P, C.c_long, C.c_int, P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


_ERR = {-1: "bad argument", -2: "expert id outside [-1, E)", -3: "padded rows exceed capacity",
        -4: "out of memory"}


def capacity(T: int, k: int, E: int, tm: int) -> int:
    """Rows that always hold the padded plan: T*k + min(E, T*k)*(tm-1)."""
    n = T * k
    return n + min(E, n) * (tm - 1)


def plan(ids, w, E: int, tm: int, cap: int | None = None) -> dict:
    """Routing plan of ids/w [T,k]: offsets, counts, srt_tok, srt_w, pos,
    tile_expert (arrays trimmed to R_pad rows / R_pad/tm tiles) and R_pad."""
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    T, k = ids.shape
    if cap is None:
        cap = capacity(T, k, E, tm)
    offsets = np.zeros(E + 1, np.int32)
    counts = np.zeros(E, np.int32)
    srt_tok = np.full(max(cap, 1), -7, np.int32)
    srt_w = np.full(max(cap, 1), np.nan, np.float32)
    pos = np.full(max(T * k, 1), -7, np.int32)
    tile_expert = np.full(max(cap // tm + 1, 1), -7, np.int32)
    r = _load().oracle_plan(_p(ids), _p(w), T, k, E, tm, _p(offsets), _p(counts),
                            _p(srt_tok), _p(srt_w), _p(pos), _p(tile_expert), cap)
    if r < 0:
        raise OracleError(_ERR.get(r, str(r)))
    return dict(R_pad=int(r), offsets=offsets, counts=counts, srt_tok=srt_tok[:r],
                srt_w=srt_w[:r], pos=pos[:T * k].reshape(T, k),
                tile_expert=tile_expert[:r // tm])


def gather(x, srt_tok) -> np.ndarray:
    """xs[r] = x[srt_tok[r]] (16-bit rows), zero rows where srt_tok is -1."""
    x = _c(x, np.uint16)
    T, d = x.shape
    srt_tok = _c(srt_tok, np.int32)
    R = srt_tok.shape[0]
    xs = np.empty((max(R, 1), d), np.uint16)
    _load().oracle_gather(_p(x), T, d, _p(srt_tok), R, _p(xs))
    return xs[:R]


def _weights(Wg, Wu, Wd):
    """bf16 bit arrays, or (E4M3 codes, fp32 scales) pairs: the arrays the C
    side takes, the shapes (E, d, f), and whether they are E4M3."""
    q8 = isinstance(Wg, tuple)
    if q8:
        (g, sg), (u, su), (dn, sd) = Wg, Wu, Wd
        g, u, dn = _c(g, np.uint8), _c(u, np.uint8), _c(dn, np.uint8)
        sg, su, sd = _c(sg, np.float32), _c(su, np.float32), _c(sd, np.float32)
        E, d, f = g.shape
        assert sg.shape == (E, f) and su.shape == (E, f) and sd.shape == (E, d)
        arrs = (g, sg, u, su, dn, sd)
    else:
        g, u, dn = _c(Wg, np.uint16), _c(Wu, np.uint16), _c(Wd, np.uint16)
        E, d, f = g.shape
        arrs = (g, u, dn)
    assert u.shape == g.shape and dn.shape == (E, f, d)
    return arrs, (E, d, f), q8


def layer(x, ids, w, Wg, Wu, Wd, x_dtype: str = "bf16", tokens=None,
          mirror: bool = False, nthreads: int | None = None, act_e4m3: bool = False) -> np.ndarray:
    """Layer output y (fp64 [len(tokens), d]) for the listed tokens (all by
    default).  ``mirror`` returns the bf16-mirror reference instead.  The
    weights are bf16 bit arrays or, all three, (E4M3 codes, scales) pairs;
    with E4M3 weights, ``act_e4m3`` gives gate/up the rows' E4M3 values
    (``quantize_rows_e4m3``)."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    warrs, (E, d2, f), q8 = _weights(Wg, Wu, Wd)
    T, d = x.shape
    k = ids.shape[1]
    assert d2 == d
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = _c(tokens, np.int32)
    y = np.zeros((max(len(tokens), 1), d), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    assert q8 or not act_e4m3, "E4M3 activations come with E4M3 weights"
    if q8:
        rc = _load().oracle_layer_tokens_e4m3(
            _p(x), int(x_dtype == "f16"), _p(ids), _p(w), *[_p(a) for a in warrs], T, d, E, k,
            f, _p(tokens), len(tokens), int(bool(mirror)), int(bool(act_e4m3)), int(nthreads),
            _p(y))
    else:
        rc = _load().oracle_layer_tokens(
            _p(x), int(x_dtype == "f16"), _p(ids), _p(w), *[_p(a) for a in warrs], T, d, E, k,
            f, _p(tokens), len(tokens), int(bool(mirror)), int(nthreads), _p(y))
    if rc != 0:
        raise OracleError(_ERR.get(rc, str(rc)))
    return y[:len(tokens)]


def expert_rows(xs, rows, row_expert, row_w, Wg, Wu, Wd, x_dtype: str = "bf16",
                mirror: bool = False, nthreads: int | None = None, act_e4m3: bool = False):
    """For the listed rows of xs: h (fp64 [n, f]) and the weighted down
    projection ys = w * o (fp64 [n, d])."""
    xs = _c(xs, np.uint16)
    d = xs.shape[1]
    warrs, (E, _, f), q8 = _weights(Wg, Wu, Wd)
    rows = _c(rows, np.int64)
    row_expert = _c(row_expert, np.int32)
    row_w = _c(row_w, np.float32)
    n = len(rows)
    h = np.zeros((max(n, 1), f), np.float64)
    ys = np.zeros((max(n, 1), d), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    assert q8 or not act_e4m3, "E4M3 activations come with E4M3 weights"
    if q8:
        rc = _load().oracle_expert_rows_e4m3(
            _p(xs), int(x_dtype == "f16"), d, f, _p(rows), n, _p(row_expert), _p(row_w), E,
            *[_p(a) for a in warrs], int(bool(mirror)), int(bool(act_e4m3)), int(nthreads),
            _p(h), _p(ys))
    else:
        rc = _load().oracle_expert_rows(
            _p(xs), int(x_dtype == "f16"), d, f, _p(rows), n, _p(row_expert), _p(row_w), E,
            *[_p(a) for a in warrs], int(bool(mirror)), int(nthreads), _p(h), _p(ys))
    if rc != 0:
        raise OracleError(_ERR.get(rc, str(rc)))
    return h[:n], ys[:n]


def combine(Ys, pos) -> np.ndarray:
    """y[t] = sum_j Ys[pos[t,j]] over j = 0..k-1 in order (fp64)."""
    Ys = _c(Ys, np.uint16)
    pos = _c(pos, np.int32)
    T, k = pos.shape
    d = Ys.shape[1]
    y = np.zeros((max(T, 1), d), np.float64)
    _load().oracle_combine(_p(Ys), _p(pos), T, k, d, _p(y))
    return y[:T]


def round_bf16(v: float) -> float:
    return _load().oracle_round_bf16(float(v))


def value16(bits: int, dtype: str = "bf16") -> float:
    return _load().oracle_value16(int(bits), int(dtype == "f16"))


def e4m3_value(code: int) -> float:
    """Value of an E4M3 code (NaN for S.1111.111)."""
    return _load().oracle_e4m3_value(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    """Nearest E4M3 code to the fp32 value v, ties to even, saturating at 448."""
    return int(_load().oracle_e4m3_encode(float(v)))


def quantize_e4m3(W):
    """bf16 weights [E, K, M] -> (E4M3 codes uint8 [E, K, M], fp32 scales
    [E, M]) with scale = max_k |W| / 448 (1 where that is 0) and code =
    e4m3_encode(W / scale)."""
    W = _c(W, np.uint16)
    E, K, M = W.shape
    q = np.empty((E, K, M), np.uint8)
    s = np.empty((E, M), np.float32)
    _load().oracle_quantize_e4m3(_p(W), E, K, M, _p(q), _p(s))
    return q, s


def dequantize_e4m3(q, s) -> np.ndarray:
    """fp64 weights e4m3_value(q) * scale (exact)."""
    table = np.array([e4m3_value(c) for c in range(256)], np.float64)
    q = np.asarray(q, np.uint8)
    return table[q] * np.asarray(s, np.float64)[:, None, :]


def e2m1_value(c: int) -> float:
    """Value of a 4-bit E2M1 code (OCP MX): 1 sign, 2 exponent bits (bias
    1), 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    return float(_load().oracle_e2m1_value(int(c) & 0xF))


def quantize_mxfp4(W):
    """bf16 weights [E, K, M] -> MXFP4 along K: (codes uint8 [E, K, M/2], two
    4-bit E2M1 codes a byte, feature m even in the low nibble; scale
    exponents uint8 [E, K/32, M], scale = 2^(S-127)).  Per block of 32 k:
    x = floor(log2(max|W|)) - 2 clamped to [-127, 127] (-127 for a zero
    block), S = x + 127, code = nearest E2M1 to W / 2^x (ties to even,
    saturated at 6).  K must be a multiple of 32, M even."""
    W = _c(W, np.uint16)
    E, K, M = W.shape
    if K % 32 or M % 2:
        raise OracleError("MXFP4 needs K % 32 == 0 and M even")
    codes = np.zeros((E, K, M // 2), np.uint8)
    scales = np.empty((E, K // 32, M), np.uint8)
    _load().oracle_quantize_mxfp4(_p(W), E, K, M, _p(codes), _p(scales))
    return codes, scales


def dequantize_mxfp4(codes, scales) -> np.ndarray:
    """The dequantized weights e2m1(code) * 2^(S-127) as bf16 bit patterns
    [E, K, M] (exact for S <= 252: every such value is a bf16 value).  The
    layer on MXFP4 weights is the bf16 layer on these weights."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    E, K, M2 = codes.shape
    W = np.empty((E, K, 2 * M2), np.uint16)
    rc = _load().oracle_dequantize_mxfp4(_p(codes), _p(scales), E, K, 2 * M2, _p(W))
    if rc != 0:
        raise OracleError("MXFP4 value outside bf16 (scale exponent above 252)")
    return W


def quantize_rows_e4m3(x):
    """bf16 rows x [R, d] -> (E4M3 codes [R, d], exponents e [R]): each row
    scaled by 2^-e, e the smallest integer with max|x| <= 448 * 2^e (0 for a
    zero row), codes the nearest E4M3 values.  value(code) * 2^e is the row
    gate/up sees with E4M3 activations."""
    x = _c(x, np.uint16)
    R, d = x.shape
    q = np.empty((max(R, 1), d), np.uint8)
    e = np.empty(max(R, 1), np.int32)
    _load().oracle_quantize_rows_e4m3(_p(x), R, d, _p(q), _p(e))
    return q[:R], e[:R]
