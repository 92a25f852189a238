"""The C ABI on the CPU: the library loads, exports every entry point the
header declares, and its host-side logic (sizes, workspace layout, argument
checks) behaves as documented.  No call here reaches the GPU: every call
either is host-only or fails its argument checks before anything is
enqueued (device pointers below are never dereferenced)."""
import ctypes as C
import os
import re

import pytest

from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_prefill.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def declared():
    src = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    names = set(declared())
    assert {"moe_plan", "moe_gather", "moe_expert_ffn", "moe_combine", "moe_layer_forward",
            "moe_ffn_gate_up", "moe_ffn_down", "moe_capacity", "moe_workspace_bytes",
            "moe_read_status", "moe_status_str"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name
        assert name in B._SIGS, f"binding lacks {name}"


def test_capacity(lib):
    assert B.capacity(2048, 10, 512, 16) == 20480 + 512 * 15
    assert B.capacity(4, 2, 512, 16) == 8 + 8 * 15
    assert B.capacity(0, 2, 5, 16) == 0
    for bad in ((-1, 2, 4, 16), (4, 0, 4, 16), (4, 2, 0, 16), (4, 2, 4097, 16), (4, 2, 4, 0),
                (4, 2, 4, 1025), (1 << 30, 4, 4, 16)):
        assert lib.moe_capacity(*bad) == -1


def test_workspace_layout(lib):
    T, d, E, k, f, tm = 2048, 2560, 512, 10, 512, 16
    L = B.workspace_layout(T, d, E, k, f, tm)
    offs = [L[n] for n in B.WS_FIELDS]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    cap = B.capacity(T, k, E, tm)
    assert L["Ys"] - L["H"] >= cap * f * 2 and L["total"] - L["Ys"] >= cap * d * 2
    assert L["xs"] - L["tile_expert"] >= (cap // tm) * 4 and L["H"] - L["xs"] >= cap * d * 2
    assert B.workspace_bytes(T, d, E, k, f, tm) == L["total"]
    assert L["bcnt"] == 256 and L["offsets"] == B.plan_workspace_bytes(T, k, E)


FAKE = 0x10000  # a 256-byte aligned stand-in device address, never dereferenced


def plan_call(lib, **kw):
    a = dict(ids=FAKE, w=FAKE, T=8, k=2, E=4, tm=16, offsets=FAKE, counts=FAKE, srt_tok=FAKE,
             srt_w=FAKE, pos=FAKE, tile=FAKE, cap=8 * 2 + 4 * 15, ws=FAKE, ws_bytes=1 << 20,
             stream=None)
    a.update(kw)
    return lib.moe_plan(a["ids"], a["w"], a["T"], a["k"], a["E"], a["tm"], a["offsets"],
                        a["counts"], a["srt_tok"], a["srt_w"], a["pos"], a["tile"], a["cap"],
                        a["ws"], a["ws_bytes"], a["stream"])


def test_plan_argument_errors(lib):
    assert plan_call(lib, ids=None) == B.MOE_ERR_NULL
    assert plan_call(lib, ws=None) == B.MOE_ERR_NULL
    assert plan_call(lib, E=0) == B.MOE_ERR_SHAPE
    assert plan_call(lib, E=5000) == B.MOE_ERR_SHAPE
    assert plan_call(lib, k=300) == B.MOE_ERR_SHAPE
    assert plan_call(lib, tm=0) == B.MOE_ERR_SHAPE
    assert plan_call(lib, cap=8 * 2 + 4 * 15 - 1) == B.MOE_ERR_CAPACITY
    assert plan_call(lib, ws_bytes=16) == B.MOE_ERR_WORKSPACE
    assert plan_call(lib, ids=FAKE + 2) == B.MOE_ERR_ALIGN
    assert plan_call(lib, ws=FAKE + 16) == B.MOE_ERR_ALIGN


def test_stage_argument_errors(lib):
    g = lib.moe_gather
    assert g(FAKE, 2, 8, 64, FAKE, FAKE, 4, 100, FAKE, None) == B.MOE_ERR_DTYPE
    assert g(FAKE, 0, 8, 60, FAKE, FAKE, 4, 100, FAKE, None) == B.MOE_ERR_SHAPE   # d % 8
    assert g(None, 0, 8, 64, FAKE, FAKE, 4, 100, FAKE, None) == B.MOE_ERR_NULL
    assert g(FAKE + 8, 0, 8, 64, FAKE, FAKE, 4, 100, FAKE, None) == B.MOE_ERR_ALIGN
    assert g(FAKE, 0, 8, 64, FAKE, FAKE, 4, 0, FAKE, None) == B.MOE_OK          # nothing to do
    gu = lib.moe_ffn_gate_up
    assert gu(FAKE, FAKE, FAKE, FAKE, 4, 96, 64, 100, FAKE, None, None) == B.MOE_ERR_SHAPE
    assert gu(FAKE, FAKE, FAKE, FAKE, 4, 64, 32, 100, FAKE, None, None) == B.MOE_ERR_SHAPE
    assert gu(FAKE, None, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert gu(FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, FAKE + 2, None) == B.MOE_ERR_ALIGN
    gr = lib.moe_ffn_gate_up_rows
    assert gr(FAKE, 8, None, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert gr(FAKE, -1, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_SHAPE
    assert gr(FAKE, 8, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 0, FAKE, None, None) == B.MOE_OK
    dn = lib.moe_ffn_down
    assert dn(FAKE, FAKE, FAKE, None, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    c = lib.moe_combine
    assert c(FAKE, FAKE, 4, 0, 64, FAKE, None) == B.MOE_ERR_SHAPE
    assert c(FAKE, FAKE, 0, 2, 64, FAKE, None) == B.MOE_OK
    assert c(None, FAKE, 4, 2, 64, FAKE, None) == B.MOE_ERR_NULL
    lf = lib.moe_layer_forward
    ws = 1 << 40
    assert lf(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 4, 2, 64, 8, FAKE, FAKE, ws, None) == B.MOE_ERR_SHAPE
    assert lf(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 4, 2, 64, 16, FAKE, FAKE, 10, None) == B.MOE_ERR_WORKSPACE
    assert lf(FAKE, FAKE, FAKE, None, FAKE, FAKE, 8, 64, 4, 2, 64, 16, FAKE, FAKE, ws, None) == B.MOE_ERR_NULL
    assert lib.moe_read_status(None, None, None) == B.MOE_ERR_NULL


def test_prefill_host_workspace(lib):
    T, d, E, k, f, tm = 4096, 2816, 128, 8, 704, 16
    layer = B.workspace_bytes(T, d, E, k, f, tm)
    up = lambda v: (v + 255) // 256 * 256
    staging = up(T * d * 2) + 2 * up(T * k * 4) + up(T * d * 2)
    assert B.prefill_host_workspace_bytes(T, d, E, k, f, tm) == up(layer) + 2 * staging
    assert B.prefill_host_workspace_bytes(T, d, 0, k, f, tm) == 0


def prefill_host_call(lib, n=2, ptrs=None, **kw):
    # host pointer arrays of stand-in addresses: only checked for NULL here
    arr = (C.c_void_p * max(n, 1))(*([FAKE] * max(n, 1)))
    a = dict(x=arr, ids=arr, w=arr, y=arr, Wg=FAKE, Wu=FAKE, Wd=FAKE, sg=None, su=None, sd=None,
             act=0, T=8, d=64, E=4, k=2, f=64, tm=16, ws=FAKE, ws_bytes=1 << 30)
    a.update(ptrs or {})
    a.update(kw)
    cast = lambda v: C.cast(v, C.c_void_p) if isinstance(v, C.Array) else v
    return lib.moe_prefill_forward_host(n, cast(a["x"]), cast(a["ids"]), cast(a["w"]),
                                        cast(a["y"]), a["Wg"], a["Wu"], a["Wd"], a["sg"],
                                        a["su"], a["sd"], a["act"], a["T"], a["d"], a["E"], a["k"],
                                        a["f"], a["tm"], a["ws"], a["ws_bytes"], None)


def test_prefill_host_argument_errors(lib):
    assert prefill_host_call(lib, n=-1) == B.MOE_ERR_SHAPE
    assert prefill_host_call(lib, tm=8) == B.MOE_ERR_SHAPE
    assert prefill_host_call(lib, d=96) == B.MOE_ERR_SHAPE
    assert prefill_host_call(lib, E=0) == B.MOE_ERR_SHAPE
    assert prefill_host_call(lib, Wd=None) == B.MOE_ERR_NULL
    assert prefill_host_call(lib, ptrs={"y": None}) == B.MOE_ERR_NULL
    holed = (C.c_void_p * 2)(FAKE, None)  # chunk 1 has no x
    assert prefill_host_call(lib, ptrs={"x": holed}) == B.MOE_ERR_NULL
    assert prefill_host_call(lib, ws_bytes=1024) == B.MOE_ERR_WORKSPACE
    assert prefill_host_call(lib, ws=FAKE + 128) == B.MOE_ERR_ALIGN
    assert prefill_host_call(lib, Wg=FAKE + 8) == B.MOE_ERR_ALIGN
    assert prefill_host_call(lib, sg=FAKE) == B.MOE_ERR_NULL      # E4M3 needs all three scales
    assert prefill_host_call(lib, act=1, d=128) == B.MOE_ERR_NULL  # E4M3 rows need E4M3 weights
    assert prefill_host_call(lib, act=1, sg=FAKE, su=FAKE, sd=FAKE, d=96) == B.MOE_ERR_SHAPE
    # nothing to do: returns before any CUDA call
    assert prefill_host_call(lib, n=0) == B.MOE_OK
    assert prefill_host_call(lib, T=0) == B.MOE_OK


def test_e4m3_argument_errors(lib):
    q = lib.moe_quantize_e4m3
    assert q(FAKE, 0, 8, 64, FAKE, FAKE, 0, None) == B.MOE_ERR_SHAPE
    assert q(FAKE, 4, 0, 64, FAKE, FAKE, 0, None) == B.MOE_ERR_SHAPE
    assert q(FAKE, 4, 96, 64, FAKE, FAKE, 1, None) == B.MOE_ERR_SHAPE    # K-major: K % 64
    assert q(None, 4, 8, 64, FAKE, FAKE, 0, None) == B.MOE_ERR_NULL
    assert q(FAKE, 4, 8, 64, FAKE, FAKE + 2, 0, None) == B.MOE_ERR_ALIGN
    g8 = lib.moe_gather_e4m3
    assert g8(FAKE, 8, 72, FAKE, FAKE, 4, 100, FAKE, FAKE, None) == B.MOE_ERR_SHAPE  # d % 16
    assert g8(FAKE, 8, 64, FAKE, FAKE, 4, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert g8(FAKE, 8, 64, FAKE, FAKE, 4, 100, FAKE + 8, FAKE, None) == B.MOE_ERR_ALIGN
    assert g8(FAKE, 8, 64, FAKE, FAKE, 4, 0, FAKE, FAKE, None) == B.MOE_OK
    gf = lib.moe_ffn_gate_up_f8
    assert gf(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 96, 64, 100, FAKE, None, None) == B.MOE_ERR_SHAPE
    assert gf(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 128, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    r8 = lib.moe_rows_e4m3
    assert r8(FAKE, 24, FAKE, 4, 100, FAKE, FAKE, None) == B.MOE_ERR_SHAPE
    assert r8(FAKE, 64, FAKE, 4, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert r8(FAKE, 64, FAKE, 4, 0, FAKE, FAKE, None) == B.MOE_OK
    df = lib.moe_ffn_down_f8
    assert df(FAKE, None, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert df(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 0, FAKE, None, None) == B.MOE_OK
    assert gf(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 128, 64, 0, FAKE, None, None) == B.MOE_OK
    gu = lib.moe_ffn_gate_up_e4m3
    assert gu(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 96, 64, 100, FAKE, None, None) == B.MOE_ERR_SHAPE
    assert gu(FAKE, FAKE, None, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert gu(FAKE, FAKE + 8, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_ALIGN
    assert gu(FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_ALIGN
    assert gu(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 0, FAKE, None, None) == B.MOE_OK
    dn = lib.moe_ffn_down_e4m3
    assert dn(FAKE, FAKE, None, FAKE, FAKE, 4, 64, 64, 100, FAKE, None, None) == B.MOE_ERR_NULL
    assert dn(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 0, FAKE, None, None) == B.MOE_OK
    lf8 = lib.moe_layer_forward_f8
    assert lf8(*([FAKE] * 9 + [8, 96, 4, 2, 64, 16, FAKE, FAKE, 1 << 40, None])) == B.MOE_ERR_SHAPE
    lf = lib.moe_layer_forward_e4m3
    ws = 1 << 40
    args = [FAKE] * 9 + [8, 64, 4, 2, 64, 16, FAKE, FAKE, ws, None]
    bad = list(args); bad[4] = None                                    # su missing
    assert lf(*bad) == B.MOE_ERR_NULL
    bad = list(args); bad[1 + 1] = FAKE + 2                             # w misaligned
    assert lf(*bad) == B.MOE_ERR_ALIGN
    bad = list(args); bad[14] = 8                                       # tm
    assert lf(*bad) == B.MOE_ERR_SHAPE


def test_moe_layer_holds_either_weight_form():
    import torch
    t = lambda *shape: torch.empty(*shape, dtype=torch.bfloat16)
    L = B.MoeLayer(t(2, 64, 128), t(2, 64, 128), t(2, 128, 64))
    assert (L.E, L.d, L.f, L.e4m3) == (2, 64, 128, False) and L._ws is None
    q = lambda *shape: (torch.empty(*shape, dtype=torch.uint8),
                        torch.empty(shape[0], shape[2], dtype=torch.float32))
    L8 = B.MoeLayer(q(2, 64, 128), q(2, 64, 128), q(2, 128, 64))
    assert (L8.E, L8.d, L8.f, L8.e4m3) == (2, 64, 128, True) and L8._host_ws is None
    # E4M3 rows: gate/up codes K-major [E, f, d]
    Lf = B.MoeLayer(q(2, 128, 64), q(2, 128, 64), q(2, 128, 64), act_e4m3=True)
    assert (Lf.E, Lf.d, Lf.f, Lf.act_e4m3) == (2, 64, 128, True)
    with pytest.raises(ValueError):
        B.MoeLayer(t(2, 64, 128), t(2, 64, 128), t(2, 128, 64), act_e4m3=True)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 99):
        assert isinstance(B.status_str(code), str) and B.status_str(code)


def test_plan_workspace_holds_block_and_group_counts(lib):
    # one row of E int32 per block of 4096 entries and one per group of 256
    # blocks, after the 256-byte header
    for T, k, E in [(1, 1, 1), (2048, 10, 512), (104858, 10, 512), (1 << 20, 10, 512),
                    (65537, 4, 4096), (70001, 2, 256)]:
        nblk = -(-(T * k) // 4096)
        rows = nblk + -(-nblk // 256)
        want = 256 + -(-(rows * E * 4) // 256) * 256
        assert B.plan_workspace_bytes(T, k, E) == want, (T, k, E)


def noalloc_call(lib, T, k, E, status):
    tm = 16
    return lib.moe_plan_noalloc(FAKE, FAKE, T, k, E, tm, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                B.capacity(T, k, E, tm), status, None)


@pytest.mark.parametrize("E,entries", [(512, 517 * 4096), (4096, 64 * 4096)])
def test_noalloc_limit_boundary(lib, E, entries):
    # (blocks + groups) x E <= MOE_PLAN_NOALLOC_MAX_COUNTS: at the limit the
    # size check passes (the misaligned status word is the first error, so
    # nothing is enqueued); one entry more needs another block row
    k = 4 if E == 4096 else 1
    T = entries // k
    assert noalloc_call(lib, T, k, E, FAKE + 2) == B.MOE_ERR_ALIGN
    T1 = (entries + k) // k
    assert noalloc_call(lib, T1, k, E, FAKE + 2) == B.MOE_ERR_WORKSPACE


def test_mxfp4_argument_checks(lib):
    FAKEP = 1 << 20
    # K a multiple of 32 and M even; null and misaligned pointers
    assert lib.moe_quantize_mxfp4(FAKEP, 2, 48, 64, FAKEP, FAKEP, None) == B.MOE_ERR_SHAPE
    assert lib.moe_quantize_mxfp4(FAKEP, 2, 64, 63, FAKEP, FAKEP, None) == B.MOE_ERR_SHAPE
    assert lib.moe_quantize_mxfp4(None, 2, 64, 64, FAKEP, FAKEP, None) == B.MOE_ERR_NULL
    assert lib.moe_quantize_mxfp4(FAKEP, 2, 64, 64, FAKEP + 8, FAKEP, None) == B.MOE_ERR_ALIGN
    assert lib.moe_quantize_mxfp4(FAKEP + 2, 2, 64, 64, FAKEP, FAKEP, None) == B.MOE_ERR_ALIGN
    # GEMMs: d and f multiples of 64, scale exponents present and 16-byte aligned
    args = (FAKEP, FAKEP, FAKEP, FAKEP, FAKEP, FAKEP)
    assert lib.moe_ffn_gate_up_mxfp4(*args, 4, 96, 64, 64, FAKEP, None, None) == B.MOE_ERR_SHAPE
    assert lib.moe_ffn_gate_up_mxfp4(FAKEP, FAKEP, None, FAKEP, FAKEP, FAKEP, 4, 64, 64, 64,
                                     FAKEP, None, None) == B.MOE_ERR_NULL
    assert lib.moe_ffn_gate_up_mxfp4(FAKEP, FAKEP, FAKEP + 8, FAKEP, FAKEP, FAKEP, 4, 64, 64, 64,
                                     FAKEP, None, None) == B.MOE_ERR_ALIGN
    assert lib.moe_ffn_down_mxfp4(FAKEP, FAKEP, None, FAKEP, FAKEP, 4, 64, 64, 64, FAKEP, None,
                                  None) == B.MOE_ERR_NULL
    assert lib.moe_layer_forward_mxfp4(FAKEP, FAKEP, FAKEP, FAKEP, None, FAKEP, FAKEP, FAKEP,
                                       FAKEP, 8, 64, 4, 2, 64, 16, FAKEP, FAKEP, 1 << 30,
                                       None) == B.MOE_ERR_NULL
