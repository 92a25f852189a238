"""Shared helpers of the tests: cached seeded inputs, host/device moves and
the layer tolerance (max|y - ref| <= 1e-2 * max|ref| + 1e-3)."""
import functools

import numpy as np
import torch

from moe_prefill_routing_gb300 import workload as W


@functools.lru_cache(maxsize=8)
def inputs(cfg, chunk: int = 0, seed: int = 0):
    """Host inputs of a named workload (cached per process)."""
    return W.make_inputs(cfg, seed=seed, chunk=chunk)


_dev_cache = {}


def dev_weights(cfg, seed: int = 0):
    """Device copies of a workload's weights (cached per process)."""
    key = (cfg, seed)
    if key not in _dev_cache:
        inp = inputs(cfg, 0, seed)
        _dev_cache[key] = tuple(dev16(inp[n]) for n in ("Wg", "Wu", "Wd"))
    return _dev_cache[key]


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def dev16(bits, dtype=torch.bfloat16, device="cuda"):
    """uint16 bit patterns -> device bf16 (or fp16) tensor, bits unchanged."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(dtype)


def host16(t):
    """Device 16-bit tensor -> uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f(t):
    """Device bf16/fp16 tensor -> float64 values."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def layer_tolerance(y, ref):
    """max|y - ref| <= 1e-2 * max|ref| + 1e-3 (bf16 operands, fp32 accumulation)."""
    err = float(np.max(np.abs(y - ref))) if y.size else 0.0
    bound = 1e-2 * (float(np.max(np.abs(ref))) if ref.size else 0.0) + 1e-3
    return err <= bound, err, bound


def rel_l2(y, ref):
    n = float(np.linalg.norm(ref))
    return float(np.linalg.norm(y - ref)) / n if n > 0 else float(np.linalg.norm(y))


def sample_tokens(ids, n, seed=0):
    """Tokens to check one by one at full size: the first and last tokens,
    tokens routed to the largest and to the smallest non-empty expert, and a
    seeded random draw."""
    T, k = ids.shape
    rng = np.random.default_rng(seed)
    flat = ids.ravel()
    valid = flat >= 0
    counts = np.bincount(flat[valid], minlength=int(flat.max()) + 1 if valid.any() else 1)
    picks = [0, T - 1]
    big = int(np.argmax(counts))
    small = int(np.argmin(np.where(counts > 0, counts, counts.max() + 1)))
    for e in (big, small):
        toks = np.nonzero((ids == e).any(axis=1))[0]
        picks += list(toks[:2]) + list(toks[-2:])
    picks += list(rng.choice(T, size=max(0, n - len(picks)), replace=False))
    out = []
    for t in picks:
        if int(t) not in out:
            out.append(int(t))
    return np.array(out[:max(n, 1)], dtype=np.int32)
