"""Thin binding of ``libmoe_prefill.so`` (the C ABI in ``include/moe_prefill.h``).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  There
is no fallback: if the library is missing or a call fails, this raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import NamedTuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_prefill.so")
_lock = threading.Lock()
_lib = None

# return codes and status bits (include/moe_prefill.h)
MOE_OK = 0
MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_CAPACITY, MOE_ERR_WORKSPACE = -1, -2, -3, -4
MOE_ERR_ALIGN, MOE_ERR_CUDA, MOE_ERR_DTYPE = -5, -6, -7
STATUS_BAD_ID, STATUS_OVERFLOW, STATUS_BAD_OFFSETS, STATUS_TIMEOUT = 1, 2, 4, 8
DT_BF16, DT_F16 = 0, 1
WS_FIELDS = ["status", "bcnt", "offsets", "counts", "srt_tok", "srt_w", "pos", "tile_expert",
             "xs", "H", "Ys", "total"]

_SIGS = {
    "moe_capacity": (C.c_int64, [C.c_int] * 4),
    "moe_plan_workspace_bytes": (C.c_size_t, [C.c_int] * 3),
    "moe_plan": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                           C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                           C.c_void_p, C.c_int64, C.c_void_p, C.c_size_t, C.c_void_p]),
    "moe_plan_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                   C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                   C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p]),
    "moe_gather": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                             C.c_int, C.c_int64, C.c_void_p, C.c_void_p]),
    "moe_ffn_gate_up": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                                  C.c_int, C.c_int, C.c_int64, C.c_void_p, C.c_void_p,
                                  C.c_void_p]),
    "moe_ffn_gate_up_rows": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int64,
                                       C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_ffn_down": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                               C.c_int, C.c_int, C.c_int64, C.c_void_p, C.c_void_p,
                               C.c_void_p]),
    "moe_expert_ffn": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                 C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int64, C.c_void_p,
                                 C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_combine": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                              C.c_void_p]),
    "moe_workspace_bytes": (C.c_size_t, [C.c_int] * 6),
    "moe_workspace_layout": (C.c_int, [C.c_int] * 6 + [C.c_void_p]),
    "moe_layer_forward": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                    C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_size_t,
                                    C.c_void_p]),
    "moe_prefill_host_workspace_bytes": (C.c_size_t, [C.c_int] * 6),
    "moe_prefill_forward_host": (C.c_int, [C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_void_p, C.c_int,
                                           C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                           C.c_void_p, C.c_size_t, C.c_void_p]),
    "moe_quantize_e4m3": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                    C.c_void_p, C.c_int, C.c_void_p]),
    "moe_gather_e4m3": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int,
                                  C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_ffn_gate_up_f8": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                     C.c_int, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_rows_e4m3": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_int64, C.c_void_p,
                                C.c_void_p, C.c_void_p]),
    "moe_ffn_down_f8": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int64, C.c_void_p,
                                  C.c_void_p, C.c_void_p]),
    "moe_layer_forward_f8": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                       C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_size_t,
                                       C.c_void_p]),
    "moe_ffn_gate_up_e4m3": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                       C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_ffn_down_e4m3": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                    C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int64,
                                    C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_layer_forward_e4m3": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                         C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_size_t,
                                         C.c_void_p]),
    "moe_quantize_mxfp4": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                     C.c_void_p, C.c_void_p]),
    "moe_ffn_gate_up_mxfp4": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                        C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_ffn_down_mxfp4": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int64,
                                     C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_layer_forward_mxfp4": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int,
                                          C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_size_t,
                                          C.c_void_p]),
    "moe_read_status": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p]),
    "moe_selftest_wait_limit": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_int, C.c_int, C.c_int, C.c_int64, C.c_void_p,
                                          C.c_void_p, C.c_int, C.c_void_p]),
    "moe_status_str": (C.c_char_p, [C.c_int]),
}


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({status_str(code)})")


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m moe_prefill_routing_gb300.build`")
            L = C.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().moe_status_str(int(code)).decode()


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(device=None) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(t) -> int:
    if t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return DT_BF16
    if t.dtype == torch.float16:
        return DT_F16
    raise ValueError(f"unsupported 16-bit dtype {t.dtype}")


# ---- sizes ----------------------------------------------------------------

def capacity(T: int, k: int, E: int, tm: int) -> int:
    c = lib().moe_capacity(T, k, E, tm)
    if c < 0:
        raise MoeError("moe_capacity", MOE_ERR_SHAPE)
    return int(c)


def plan_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(lib().moe_plan_workspace_bytes(T, k, E))


def workspace_bytes(T: int, d: int, E: int, k: int, f: int, tm: int) -> int:
    return int(lib().moe_workspace_bytes(T, d, E, k, f, tm))


def workspace_layout(T: int, d: int, E: int, k: int, f: int, tm: int) -> dict:
    out = (C.c_size_t * len(WS_FIELDS))()
    _check("moe_workspace_layout", lib().moe_workspace_layout(T, d, E, k, f, tm, out))
    return {name: int(out[i]) for i, name in enumerate(WS_FIELDS)}


# ---- stages ---------------------------------------------------------------

def plan(ids, w, E: int, tm: int, cap: int | None = None, out: dict | None = None) -> dict:
    """moe_plan on device tensors ids int32 [T,k], w fp32 [T,k].

    Returns the output tensors (full capacity; rows >= R_pad unwritten) and
    the plan workspace ``ws`` (status word at byte 0)."""
    T, k = ids.shape
    dev = ids.device
    if cap is None:
        cap = capacity(T, k, E, tm)
    if out is None:
        out = {}
    o = dict(out)
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("srt_tok", torch.empty(max(cap, 1), dtype=torch.int32, device=dev))
    o.setdefault("srt_w", torch.empty(max(cap, 1), dtype=torch.float32, device=dev))
    o.setdefault("pos", torch.empty((T, k), dtype=torch.int32, device=dev))
    o.setdefault("tile_expert", torch.empty(max(cap // tm, 1), dtype=torch.int32, device=dev))
    wsb = plan_workspace_bytes(T, k, E)
    o.setdefault("ws", torch.empty(wsb, dtype=torch.uint8, device=dev))
    with torch.cuda.device(dev):
        rc = lib().moe_plan(_ptr(ids), _ptr(w), T, k, E, tm, _ptr(o["offsets"]),
                            _ptr(o["counts"]), _ptr(o["srt_tok"]), _ptr(o["srt_w"]),
                            _ptr(o["pos"]), _ptr(o["tile_expert"]), cap, _ptr(o["ws"]),
                            o["ws"].numel(), _stream(dev))
    _check("moe_plan", rc)
    o["cap"] = cap
    return o


def plan_noalloc(ids, w, E: int, tm: int, cap: int | None = None, out: dict | None = None,
                 status=None) -> dict:
    """moe_plan_noalloc: the same plan as ``plan`` with the library's own
    scratch instead of a workspace (for callers that cannot allocate device
    memory).  Output tensors are allocated here only when ``out`` lacks
    them; ``status`` is an optional int32 device tensor of one element."""
    T, k = ids.shape
    dev = ids.device
    if cap is None:
        cap = capacity(T, k, E, tm)
    o = dict(out or {})
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("srt_tok", torch.empty(max(cap, 1), dtype=torch.int32, device=dev))
    o.setdefault("srt_w", torch.empty(max(cap, 1), dtype=torch.float32, device=dev))
    o.setdefault("pos", torch.empty((T, k), dtype=torch.int32, device=dev))
    o.setdefault("tile_expert", torch.empty(max(cap // tm, 1), dtype=torch.int32, device=dev))
    with torch.cuda.device(dev):
        rc = lib().moe_plan_noalloc(_ptr(ids), _ptr(w), T, k, E, tm, _ptr(o["offsets"]),
                                    _ptr(o["counts"]), _ptr(o["srt_tok"]), _ptr(o["srt_w"]),
                                    _ptr(o["pos"]), _ptr(o["tile_expert"]), cap, _ptr(status),
                                    _stream(dev))
    _check("moe_plan_noalloc", rc)
    o["cap"] = cap
    return o


def gather(x, srt_tok, offsets, E: int, cap: int, xs=None):
    """moe_gather: xs [cap, d] (16-bit) from x [T, d]."""
    T, d = x.shape
    if xs is None:
        xs = torch.empty((max(cap, 1), d), dtype=x.dtype, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().moe_gather(_ptr(x), _dtype_code(x), T, d, _ptr(srt_tok), _ptr(offsets), E,
                              cap, _ptr(xs), _stream(x.device))
    _check("moe_gather", rc)
    return xs


def ffn_gate_up(xs, Wg, Wu, offsets, cap: int, H=None, status=None):
    E, d, f = Wg.shape
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=xs.device)
    with torch.cuda.device(xs.device):
        rc = lib().moe_ffn_gate_up(_ptr(xs), _ptr(Wg), _ptr(Wu), _ptr(offsets), E, d, f, cap,
                                   _ptr(H), _ptr(status), _stream(xs.device))
    _check("moe_ffn_gate_up", rc)
    return H


def ffn_gate_up_rows(x, srt_tok, Wg, Wu, offsets, cap: int, H=None, status=None):
    """gate/up with the routed rows read from x [T, d] by srt_tok (no xs)."""
    T = x.shape[0]
    E, d, f = Wg.shape
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().moe_ffn_gate_up_rows(_ptr(x), T, _ptr(srt_tok), _ptr(Wg), _ptr(Wu),
                                        _ptr(offsets), E, d, f, cap, _ptr(H), _ptr(status),
                                        _stream(x.device))
    _check("moe_ffn_gate_up_rows", rc)
    return H


def ffn_down(H, Wd, offsets, srt_w, cap: int, Ys=None, status=None):
    E, f, d = Wd.shape
    if Ys is None:
        Ys = torch.empty((max(cap, 1), d), dtype=torch.bfloat16, device=H.device)
    with torch.cuda.device(H.device):
        rc = lib().moe_ffn_down(_ptr(H), _ptr(Wd), _ptr(offsets), _ptr(srt_w), E, d, f, cap,
                                _ptr(Ys), _ptr(status), _stream(H.device))
    _check("moe_ffn_down", rc)
    return Ys


def expert_ffn(xs, Wg, Wu, Wd, offsets, srt_w, cap: int, H=None, Ys=None, status=None):
    E, d, f = Wg.shape
    dev = xs.device
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=dev)
    if Ys is None:
        Ys = torch.empty((max(cap, 1), d), dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        rc = lib().moe_expert_ffn(_ptr(xs), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(offsets),
                                  _ptr(srt_w), E, d, f, cap, _ptr(H), _ptr(Ys), _ptr(status),
                                  _stream(dev))
    _check("moe_expert_ffn", rc)
    return H, Ys


def combine(Ys, pos, y=None):
    T, k = pos.shape
    d = Ys.shape[1]
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=Ys.device)
    with torch.cuda.device(Ys.device):
        rc = lib().moe_combine(_ptr(Ys), _ptr(pos), T, k, d, _ptr(y), _stream(Ys.device))
    _check("moe_combine", rc)
    return y


def layer_forward(x, ids, w, Wg, Wu, Wd, tm: int, y=None, ws=None):
    """moe_layer_forward: y [T, d] bf16.  ``ws`` (uint8 device tensor of
    workspace_bytes(...)) may be passed in to reuse it and to inspect the
    intermediates through workspace_layout(...)."""
    T, d = x.shape
    k = ids.shape[1]
    E, _, f = Wg.shape
    dev = x.device
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    nbytes = workspace_bytes(T, d, E, k, f, tm)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib().moe_layer_forward(_ptr(x), _ptr(ids), _ptr(w), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                     T, d, E, k, f, tm, _ptr(y), _ptr(ws), ws.numel(),
                                     _stream(dev))
    _check("moe_layer_forward", rc)
    return y


def prefill_host_workspace_bytes(T: int, d: int, E: int, k: int, f: int, tm: int) -> int:
    return lib().moe_prefill_host_workspace_bytes(T, d, E, k, f, tm)


def _host_ptrs(ts, name):
    for t in ts:
        if t.is_cuda:
            raise ValueError(f"{name}: host tensors expected")
        if not t.is_contiguous():
            raise ValueError(f"{name}: contiguous tensors expected")
    return (C.c_void_p * max(len(ts), 1))(*[t.data_ptr() for t in ts])


def prefill_forward_host(x_hs, ids_hs, w_hs, y_hs, Wg, Wu, Wd, tm: int, ws=None,
                         act_e4m3: bool = False):
    """moe_prefill_forward_host over len(x_hs) chunks: host (preferably
    pinned) x [T, d] bf16, ids/w [T, k] in; host y [T, d] bf16 out.  The
    weights are bf16 tensors or, all three, (E4M3 codes, scales) pairs.
    Asynchronous on the current stream; synchronize before reading y_hs."""
    n = len(x_hs)
    if not (len(ids_hs) == len(w_hs) == len(y_hs) == n):
        raise ValueError("one ids, w and y per chunk")
    (Wg, Wu, Wd), scales = _split_weights(Wg, Wu, Wd)
    E, f, d = Wg.shape if act_e4m3 else Wd.shape
    T, k = (ids_hs[0].shape if n else (0, 1))
    dev = Wg.device
    nbytes = prefill_host_workspace_bytes(T, d, E, k, f, tm)
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    arrays = [_host_ptrs(x_hs, "x"), _host_ptrs(ids_hs, "ids"), _host_ptrs(w_hs, "w"),
              _host_ptrs(y_hs, "y")]
    with torch.cuda.device(dev):
        rc = lib().moe_prefill_forward_host(n, *[C.cast(a, C.c_void_p) for a in arrays],
                                            _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                            *[_ptr(t) for t in scales], int(act_e4m3), T, d, E,
                                            k, f, tm,
                                            _ptr(ws), ws.numel(), _stream(dev))
    _check("moe_prefill_forward_host", rc)
    return y_hs


def _split_weights(Wg, Wu, Wd):
    """(codes, scales) pairs -> the code tensors and the scale tensors;
    bf16 tensors -> themselves and three Nones."""
    if isinstance(Wg, tuple):
        return (Wg[0], Wu[0], Wd[0]), (Wg[1], Wu[1], Wd[1])
    return (Wg, Wu, Wd), (None, None, None)


def quantize_e4m3(W, kmajor: bool = False):
    """moe_quantize_e4m3: bf16 W [E, K, M] -> (uint8 codes [E, K, M], or
    [E, M, K] with kmajor, fp32 scales [E, M]), the pair the *_e4m3 / *_f8
    calls and MoeLayer take."""
    E, K, M = W.shape
    q = torch.empty((E, M, K) if kmajor else (E, K, M), dtype=torch.uint8, device=W.device)
    s = torch.empty((E, M), dtype=torch.float32, device=W.device)
    with torch.cuda.device(W.device):
        rc = lib().moe_quantize_e4m3(_ptr(W), E, K, M, _ptr(q), _ptr(s), int(kmajor),
                                     _stream(W.device))
    _check("moe_quantize_e4m3", rc)
    return q, s


def gather_e4m3(x, srt_tok, offsets, E: int, cap: int, xs8=None, xexp=None):
    """moe_gather_e4m3: (uint8 codes [cap, d], int32 row exponents [cap])."""
    T, d = x.shape
    if xs8 is None:
        xs8 = torch.empty((max(cap, 1), d), dtype=torch.uint8, device=x.device)
    if xexp is None:
        xexp = torch.empty(max(cap, 1), dtype=torch.int32, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().moe_gather_e4m3(_ptr(x), T, d, _ptr(srt_tok), _ptr(offsets), E, cap,
                                   _ptr(xs8), _ptr(xexp), _stream(x.device))
    _check("moe_gather_e4m3", rc)
    return xs8, xexp


def ffn_gate_up_f8(xs8, xexp, Wg, Wu, offsets, cap: int, H=None, status=None):
    """moe_ffn_gate_up_f8 with K-major (codes, scales) pairs Wg, Wu [E, f, d]."""
    (qg, sg), (qu, su) = Wg, Wu
    E, f, d = qg.shape
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=xs8.device)
    with torch.cuda.device(xs8.device):
        rc = lib().moe_ffn_gate_up_f8(_ptr(xs8), _ptr(xexp), _ptr(qg), _ptr(sg), _ptr(qu),
                                      _ptr(su), _ptr(offsets), E, d, f, cap, _ptr(H),
                                      _ptr(status), _stream(xs8.device))
    _check("moe_ffn_gate_up_f8", rc)
    return H


def rows_e4m3(H, offsets, E: int, cap: int, H8=None, hexp=None):
    """moe_rows_e4m3: the rows of H [cap, f] as (uint8 codes [cap, f], int32
    exponents [cap])."""
    f = H.shape[1]
    if H8 is None:
        H8 = torch.empty((max(cap, 1), f), dtype=torch.uint8, device=H.device)
    if hexp is None:
        hexp = torch.empty(max(cap, 1), dtype=torch.int32, device=H.device)
    with torch.cuda.device(H.device):
        rc = lib().moe_rows_e4m3(_ptr(H), f, _ptr(offsets), E, cap, _ptr(H8), _ptr(hexp),
                                 _stream(H.device))
    _check("moe_rows_e4m3", rc)
    return H8, hexp


def ffn_down_f8(H8, hexp, Wd, offsets, srt_w, cap: int, Ys=None, status=None):
    """moe_ffn_down_f8 with the K-major (codes, scales) pair Wd [E, d, f]."""
    qd, sd = Wd
    E, d, f = qd.shape
    if Ys is None:
        Ys = torch.empty((max(cap, 1), d), dtype=torch.bfloat16, device=H8.device)
    with torch.cuda.device(H8.device):
        rc = lib().moe_ffn_down_f8(_ptr(H8), _ptr(hexp), _ptr(qd), _ptr(sd), _ptr(offsets),
                                   _ptr(srt_w), E, d, f, cap, _ptr(Ys), _ptr(status),
                                   _stream(H8.device))
    _check("moe_ffn_down_f8", rc)
    return Ys


def ffn_gate_up_e4m3(xs, Wg, Wu, offsets, cap: int, H=None, status=None):
    (qg, sg), (qu, su) = Wg, Wu
    E, d, f = qg.shape
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=xs.device)
    with torch.cuda.device(xs.device):
        rc = lib().moe_ffn_gate_up_e4m3(_ptr(xs), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su),
                                        _ptr(offsets), E, d, f, cap, _ptr(H), _ptr(status),
                                        _stream(xs.device))
    _check("moe_ffn_gate_up_e4m3", rc)
    return H


def ffn_down_e4m3(H, Wd, offsets, srt_w, cap: int, Ys=None, status=None):
    qd, sd = Wd
    E, f, d = qd.shape
    if Ys is None:
        Ys = torch.empty((max(cap, 1), d), dtype=torch.bfloat16, device=H.device)
    with torch.cuda.device(H.device):
        rc = lib().moe_ffn_down_e4m3(_ptr(H), _ptr(qd), _ptr(sd), _ptr(offsets), _ptr(srt_w), E,
                                     d, f, cap, _ptr(Ys), _ptr(status), _stream(H.device))
    _check("moe_ffn_down_e4m3", rc)
    return Ys


def layer_forward_e4m3(x, ids, w, Wg, Wu, Wd, tm: int, y=None, ws=None, act_e4m3: bool = False):
    """moe_layer_forward_e4m3 with (codes, scales) weight pairs, or with
    act_e4m3 moe_layer_forward_f8 (all three codes K-major)."""
    T, d = x.shape
    k = ids.shape[1]
    (qg, sg), (qu, su), (qd, sd) = Wg, Wu, Wd
    E, f = qg.shape[0], sg.shape[1]
    dev = x.device
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.empty(workspace_bytes(T, d, E, k, f, tm), dtype=torch.uint8, device=dev)
    name = "moe_layer_forward_f8" if act_e4m3 else "moe_layer_forward_e4m3"
    with torch.cuda.device(dev):
        rc = getattr(lib(), name)(_ptr(x), _ptr(ids), _ptr(w), _ptr(qg), _ptr(sg), _ptr(qu),
                                  _ptr(su), _ptr(qd), _ptr(sd), T, d, E, k, f, tm, _ptr(y),
                                  _ptr(ws), ws.numel(), _stream(dev))
    _check(name, rc)
    return y


class Mxfp4(NamedTuple):
    """MXFP4 weights of one projection: codes uint8 [E, M, K/2] (4-bit E2M1
    codes along K, eight to a 32-bit word: k = 8i + 2j at bits 4j.., its odd
    neighbour 16 bits higher) and scale
    exponents uint8 [E, K/32, M] (scale 2^(S-127) per block of 32 along K)."""
    codes: torch.Tensor
    scales: torch.Tensor


def quantize_mxfp4(W) -> Mxfp4:
    """moe_quantize_mxfp4: bf16 W [E, K, M] -> Mxfp4(codes, scales)."""
    E, K, M = W.shape
    codes = torch.empty((E, M, K // 2), dtype=torch.uint8, device=W.device)
    scales = torch.empty((E, K // 32, M), dtype=torch.uint8, device=W.device)
    with torch.cuda.device(W.device):
        rc = lib().moe_quantize_mxfp4(_ptr(W), E, K, M, _ptr(codes), _ptr(scales),
                                      _stream(W.device))
    _check("moe_quantize_mxfp4", rc)
    return Mxfp4(codes, scales)


def ffn_gate_up_mxfp4(xs, Wg: Mxfp4, Wu: Mxfp4, offsets, cap: int, H=None, status=None):
    E, f, d2 = Wg.codes.shape
    d = 2 * d2
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=xs.device)
    with torch.cuda.device(xs.device):
        rc = lib().moe_ffn_gate_up_mxfp4(_ptr(xs), _ptr(Wg.codes), _ptr(Wg.scales),
                                         _ptr(Wu.codes), _ptr(Wu.scales), _ptr(offsets), E, d, f,
                                         cap, _ptr(H), _ptr(status), _stream(xs.device))
    _check("moe_ffn_gate_up_mxfp4", rc)
    return H


def ffn_down_mxfp4(H, Wd: Mxfp4, offsets, srt_w, cap: int, Ys=None, status=None):
    E, d, f2 = Wd.codes.shape
    f = 2 * f2
    if Ys is None:
        Ys = torch.empty((max(cap, 1), d), dtype=torch.bfloat16, device=H.device)
    with torch.cuda.device(H.device):
        rc = lib().moe_ffn_down_mxfp4(_ptr(H), _ptr(Wd.codes), _ptr(Wd.scales), _ptr(offsets),
                                      _ptr(srt_w), E, d, f, cap, _ptr(Ys), _ptr(status),
                                      _stream(H.device))
    _check("moe_ffn_down_mxfp4", rc)
    return Ys


def layer_forward_mxfp4(x, ids, w, Wg: Mxfp4, Wu: Mxfp4, Wd: Mxfp4, tm: int, y=None, ws=None):
    """moe_layer_forward_mxfp4 with MXFP4 weights."""
    T, d = x.shape
    k = ids.shape[1]
    E, f = Wg.codes.shape[0], Wg.scales.shape[2]
    dev = x.device
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.empty(workspace_bytes(T, d, E, k, f, tm), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib().moe_layer_forward_mxfp4(_ptr(x), _ptr(ids), _ptr(w), _ptr(Wg.codes),
                                           _ptr(Wg.scales), _ptr(Wu.codes), _ptr(Wu.scales),
                                           _ptr(Wd.codes), _ptr(Wd.scales), T, d, E, k, f, tm,
                                           _ptr(y), _ptr(ws), ws.numel(), _stream(dev))
    _check("moe_layer_forward_mxfp4", rc)
    return y


def selftest_wait_limit(xs, Wg, Wu, offsets, cap: int, status, cta: int = 0, H=None):
    """Gate/up GEMM with CTA `cta` made to wait for bytes that never come:
    its bounded waits run out, it stops, and `status` gets STATUS_TIMEOUT."""
    E, d, f = Wg.shape
    if H is None:
        H = torch.empty((max(cap, 1), f), dtype=torch.bfloat16, device=xs.device)
    with torch.cuda.device(xs.device):
        rc = lib().moe_selftest_wait_limit(_ptr(xs), _ptr(Wg), _ptr(Wu), _ptr(offsets), E, d, f,
                                           cap, _ptr(H), _ptr(status), int(cta),
                                           _stream(xs.device))
    _check("moe_selftest_wait_limit", rc)
    return H


def read_status(ws) -> int:
    """Status word at byte 0 of a plan or layer workspace (syncs the stream)."""
    v = C.c_uint32(0)
    with torch.cuda.device(ws.device):
        rc = lib().moe_read_status(_ptr(ws), _stream(ws.device), C.byref(v))
    _check("moe_read_status", rc)
    return int(v.value)


class MoeLayer:
    """A routed MoE layer with its expert weights resident in HBM.

    The weights are bf16 tensors or, all three, (E4M3 codes, fp32 scales)
    pairs from ``quantize_e4m3`` (``MoeLayer.quantized`` makes them), or, all
    three, ``Mxfp4`` weights from ``quantize_mxfp4``
    (``MoeLayer.quantized_mxfp4``).
    ``forward`` takes device inputs.  ``forward_host`` (one chunk) and
    ``forward_host_chunks`` (a sequence of chunks) take pinned host inputs
    and go through moe_prefill_forward_host: the inputs are copied in and y
    copied back on the library's copy streams, overlapped with the layer,
    which runs on the current stream."""

    def __init__(self, Wg, Wu, Wd, tm: int = 16, act_e4m3: bool = False):
        self.Wg, self.Wu, self.Wd, self.tm = Wg, Wu, Wd, tm
        self.mxfp4 = isinstance(Wg, Mxfp4)
        if self.mxfp4:
            if act_e4m3 or not (isinstance(Wu, Mxfp4) and isinstance(Wd, Mxfp4)):
                raise ValueError("MXFP4 weights: all three projections, bf16 activations")
            self.tm, self.act_e4m3, self.e4m3 = tm, False, False
            # Wd codes [E, d, f/2]
            self.E, self.d = Wd.codes.shape[0], Wd.codes.shape[1]
            self.f = 2 * Wd.codes.shape[2]
            self.device = Wd.codes.device
            self._ws = None
            self._host_ws = None
            return
        self.e4m3 = isinstance(Wg, tuple)
        self.act_e4m3 = bool(act_e4m3)
        if self.act_e4m3 and not self.e4m3:
            raise ValueError("E4M3 activations come with E4M3 weights")
        # Wd is [E, f, d] except with E4M3 rows, where Wg is (K-major)
        ref = Wg[0] if self.act_e4m3 else (Wd[0] if self.e4m3 else Wd)
        self.E, self.f, self.d = ref.shape
        self.device = ref.device
        self._ws = None
        self._host_ws = None

    @classmethod
    def quantized(cls, Wg, Wu, Wd, tm: int = 16, act_e4m3: bool = False):
        """The same layer with its bf16 weights quantized to E4M3 on the device;
        with act_e4m3 the gate/up projection also runs on E4M3 rows (its
        weight codes K-major)."""
        return cls(quantize_e4m3(Wg, kmajor=act_e4m3), quantize_e4m3(Wu, kmajor=act_e4m3),
                   quantize_e4m3(Wd, kmajor=act_e4m3), tm=tm, act_e4m3=act_e4m3)

    @classmethod
    def quantized_mxfp4(cls, Wg, Wu, Wd, tm: int = 16):
        """The same layer with its bf16 weights quantized to MXFP4 on the device."""
        return cls(quantize_mxfp4(Wg), quantize_mxfp4(Wu), quantize_mxfp4(Wd), tm=tm)

    def workspace(self, T: int, k: int):
        n = workspace_bytes(T, self.d, self.E, k, self.f, self.tm)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x, ids, w, y=None):
        T = x.shape[0]
        ws = self.workspace(T, ids.shape[1])
        if self.mxfp4:
            return layer_forward_mxfp4(x, ids, w, self.Wg, self.Wu, self.Wd, self.tm, y=y, ws=ws)
        if self.e4m3:
            return layer_forward_e4m3(x, ids, w, self.Wg, self.Wu, self.Wd, self.tm, y=y, ws=ws,
                                      act_e4m3=self.act_e4m3)
        return layer_forward(x, ids, w, self.Wg, self.Wu, self.Wd, self.tm, y=y, ws=ws)

    def forward_host(self, x_h, ids_h, w_h, y_h):
        """Host (pinned) x, ids, w in; host y out, through the C ABI's host
        entry point.  Asynchronous on the current stream; synchronize before
        reading y_h."""
        return self.forward_host_chunks([x_h], [ids_h], [w_h], [y_h])[0]

    def forward_host_chunks(self, x_hs, ids_hs, w_hs, y_hs):
        """A sequence of prefill chunks of equal T from host memory: chunk
        c+1's inputs are copied in and chunk c-1's y copied out while chunk
        c runs.  Asynchronous on the current stream.  (The host entry point
        takes bf16 or E4M3 weights; an MXFP4 layer runs through ``forward``.)"""
        if self.mxfp4:
            raise ValueError("moe_prefill_forward_host takes bf16 or E4M3 weights, not MXFP4")
        T, k = ids_hs[0].shape
        n = prefill_host_workspace_bytes(T, self.d, self.E, k, self.f, self.tm)
        if self._host_ws is None or self._host_ws.numel() < n:
            self._host_ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        return prefill_forward_host(x_hs, ids_hs, w_hs, y_hs, self.Wg, self.Wu, self.Wd, self.tm,
                                    ws=self._host_ws, act_e4m3=self.act_e4m3)
