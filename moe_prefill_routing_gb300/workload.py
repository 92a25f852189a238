"""Seeded synthetic inputs for the routed MoE prefill layer.

This module only *draws* inputs: token activations, router choices and expert
weights.  It holds none of the layer's arithmetic (no plan, no gather, no
expert FFN, no combine), so that the CPU oracle and the CUDA path can both be
fed from it without sharing any of the method.

Recipe (every workload, seed 0 unless a test says otherwise):

* Gaussian tensors are drawn in fp32 from a torch CPU generator seeded per
  tensor from ``SeedSequence([seed, tag, chunk])``; 16-bit tensors are then
  rounded to bf16 (or fp16) with round-to-nearest-even and kept as raw
  ``uint16`` bit patterns.
* ``x ~ N(0, 1)``; ``Wg, Wu ~ N(0, 0.02)`` with layout ``[E, d, f]``;
  ``Wd ~ N(0, 0.02)`` with layout ``[E, f, d]``.
* Routing ``topk``: logits ``N(0,1)[T,E]`` (plus a per-expert bias
  ``N(0,1)[E]`` for ``topk_bias``), the k largest logits in descending order
  (ties to the lower id), weights = fp32 softmax over the chosen k.
* Routing ``zipf``: expert popularity proportional to ``rank^-1.2`` with the
  rank a seeded permutation of the ids; each token draws k distinct experts
  without replacement (Gumbel-top-k on log-popularity, slot order = draw
  order); weights = fp32 softmax of fresh ``N(0,1)`` logits over the k.

The layer shapes follow the pages: the page-1 prefill plan shape (T=2048,
E=512, top-10, tm=16, d=2560) from "Round 4 Track C: Prefill MoE Plan",
section 2, Table 2.1, plus a tiny layer, a 256-expert layer and a long-prompt
layer processed in chunks.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "workload", "make_inputs", "make_routing",
    "make_layer", "bf16_bits", "f16_bits", "bits_to_float",
]


@dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens in one layer call (a prefill chunk)
    d: int            # model width
    E: int            # experts
    k: int            # experts per token
    f: int            # expert FFN width (0: plan + gather only)
    tm: int           # tile height each expert is padded to
    x_dtype: str      # "bf16" or "f16"
    routing: str      # "topk", "topk_bias" or "zipf"
    n_chunks: int = 1  # layer calls that make up the whole prompt

    @property
    def ffn(self) -> bool:
        return self.f > 0

    @property
    def rows(self) -> int:
        return self.T * self.k


WORKLOADS = {
    1: Workload("tiny_t64_e16", T=64, d=128, E=16, k=2, f=64, tm=16,
                x_dtype="bf16", routing="topk"),
    2: Workload("plan_gather_t2048_e512_k10", T=2048, d=2560, E=512, k=10, f=0,
                tm=16, x_dtype="f16", routing="topk_bias"),
    3: Workload("layer_t2048_d2560_e512_k10_f512", T=2048, d=2560, E=512, k=10,
                f=512, tm=16, x_dtype="bf16", routing="topk_bias"),
    4: Workload("layer_t512_d4096_e256_k8_f2048", T=512, d=4096, E=256, k=8,
                f=2048, tm=16, x_dtype="bf16", routing="topk"),
    5: Workload("long_prompt_t32768_chunk4096_d2816_e128_k8_f704", T=4096,
                d=2816, E=128, k=8, f=704, tm=16, x_dtype="bf16",
                routing="zipf", n_chunks=8),
}

_TAGS = {"x": 1, "Wg": 2, "Wu": 3, "Wd": 4, "logits": 5, "bias": 6,
         "wlogits": 7, "gumbel": 8, "perm": 9, "skip": 10}


def workload(key) -> Workload:
    if isinstance(key, Workload):
        return key
    return WORKLOADS[int(key)]


def _seed(seed: int, tag: str, chunk: int = 0) -> int:
    ss = np.random.SeedSequence([int(seed), _TAGS[tag], int(chunk)])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFF_FFFF_FFFF_FFFF)


def _gen(seed: int, tag: str, chunk: int = 0) -> torch.Generator:
    return torch.Generator().manual_seed(_seed(seed, tag, chunk))


def _np_rng(seed: int, tag: str, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(_seed(seed, tag, chunk)))


def bf16_bits(a) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (round to nearest even), uint16."""
    t = torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f16_bits(a) -> np.ndarray:
    """fp32 values -> IEEE half bit patterns (round to nearest even), uint16."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def bits_to_float(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> exact fp32 values (widening is exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    raise ValueError(dtype)


def _normal16(seed, tag, shape, std, dtype, chunk=0) -> np.ndarray:
    """N(0, std) in fp32 from a per-tensor generator, rounded to 16 bits.

    Drawn one leading slice at a time so that a [E, d, f] weight never needs
    a full fp32 copy in host memory."""
    g = _gen(seed, tag, chunk)
    out = np.empty(shape, dtype=np.uint16)
    lead = shape[0] if len(shape) == 3 else 1
    sub = shape[1:] if len(shape) == 3 else shape
    conv = torch.bfloat16 if dtype == "bf16" else torch.float16
    for i in range(lead):
        t = torch.empty(sub, dtype=torch.float32).normal_(0.0, std, generator=g)
        bits = t.to(conv).view(torch.int16).numpy().view(np.uint16)
        if len(shape) == 3:
            out[i] = bits
        else:
            out[...] = bits
    return out


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float32)
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m, dtype=np.float32)
    return (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def make_routing(T: int, E: int, k: int, routing: str, seed: int = 0, chunk: int = 0):
    """Router choices for T tokens: ids int32 [T,k] and weights fp32 [T,k].

    Slot 0 holds the strongest choice.  This is input generation; the layer
    under test takes ids and weights as given."""
    if routing in ("topk", "topk_bias"):
        logits = torch.empty((T, E), dtype=torch.float32).normal_(
            0.0, 1.0, generator=_gen(seed, "logits", chunk)).numpy()
        if routing == "topk_bias":
            bias = torch.empty((E,), dtype=torch.float32).normal_(
                0.0, 1.0, generator=_gen(seed, "bias", 0)).numpy()
            logits = (logits + bias[None, :]).astype(np.float32)
        order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        ids = order.astype(np.int32)
        chosen = np.take_along_axis(logits, order, axis=1)
        w = _softmax_rows(chosen)
    elif routing == "zipf":
        perm = _np_rng(seed, "perm", 0).permutation(E)
        rank = np.empty(E, dtype=np.float64)
        rank[perm] = np.arange(1, E + 1, dtype=np.float64)
        logp = -1.2 * np.log(rank)
        u = _np_rng(seed, "gumbel", chunk).random((T, E))
        u = np.clip(u, 1e-300, 1.0 - 1e-16)
        key = logp[None, :] - np.log(-np.log(u))
        ids = np.argsort(-key, axis=1, kind="stable")[:, :k].astype(np.int32)
        wl = torch.empty((T, k), dtype=torch.float32).normal_(
            0.0, 1.0, generator=_gen(seed, "wlogits", chunk)).numpy()
        w = _softmax_rows(wl)
    else:
        raise ValueError(routing)
    return np.ascontiguousarray(ids), np.ascontiguousarray(w)


def make_inputs(wl, seed: int = 0, chunk: int = 0, weights: bool = True) -> dict:
    """All inputs of one layer call of a named workload.

    Returns a dict with ``x`` (uint16 [T,d]), ``ids`` (int32 [T,k]), ``w``
    (fp32 [T,k]) and, for FFN workloads when ``weights`` is set, ``Wg``,
    ``Wu`` (uint16 [E,d,f]) and ``Wd`` (uint16 [E,f,d]).  Weights do not
    depend on ``chunk``; activations and routing do."""
    wl = workload(wl)
    out = dict(shape=wl, seed=seed, chunk=chunk)
    out["x"] = _normal16(seed, "x", (wl.T, wl.d), 1.0, wl.x_dtype, chunk)
    out["ids"], out["w"] = make_routing(wl.T, wl.E, wl.k, wl.routing, seed, chunk)
    if wl.ffn and weights:
        out.update(make_weights(wl, seed))
    return out


def make_weights(wl, seed: int = 0) -> dict:
    wl = workload(wl)
    return dict(
        Wg=_normal16(seed, "Wg", (wl.E, wl.d, wl.f), 0.02, "bf16"),
        Wu=_normal16(seed, "Wu", (wl.E, wl.d, wl.f), 0.02, "bf16"),
        Wd=_normal16(seed, "Wd", (wl.E, wl.f, wl.d), 0.02, "bf16"),
    )


def make_layer(T: int, d: int, E: int, k: int, f: int, tm: int = 16, seed: int = 0,
               routing: str = "topk", x_dtype: str = "bf16", skip_frac: float = 0.0,
               weights: bool = True) -> dict:
    """Inputs for an arbitrary layer shape (edge-case tests).

    ``skip_frac`` marks that fraction of (token, slot) entries as skipped
    (id -1), drawn at random; the rest keep their routed expert."""
    wl = Workload(f"custom_t{T}_d{d}_e{E}_k{k}_f{f}_tm{tm}", T=T, d=d, E=E, k=k,
                  f=f, tm=tm, x_dtype=x_dtype, routing=routing)
    if k > E and routing != "zipf":
        raise ValueError("top-k routing needs k <= E")
    out = make_inputs(wl, seed=seed, weights=weights)
    if skip_frac > 0.0:
        m = _np_rng(seed, "skip", 0).random((T, k)) < skip_frac
        out["ids"] = np.where(m, -1, out["ids"]).astype(np.int32)
    return out


def with_tm(wl, tm: int) -> Workload:
    return replace(workload(wl), tm=tm)
