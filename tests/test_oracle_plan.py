"""Pins of the oracle's routing plan, gather and capacity (CPU only).

The plan is a stable counting sort ("Round 4 Track C: Prefill MoE Plan ...",
section 1 items 1-2).  It is pinned here against things other than itself:
hand-worked fixtures, a brute-force comparison sort on tiny inputs, every id
pattern of a tiny shape, and the plan's invariants on the named workloads.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from moe_prefill_routing_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_plan(ids, w, E, tm):
    """Comparison sort of the flat entries by (expert, flat index), laid out
    expert by expert with each expert's rows padded up to a multiple of tm."""
    T, k = ids.shape
    flat = [int(v) for v in ids.ravel()]
    wf = [float(v) for v in np.asarray(w, np.float32).ravel()]
    order = sorted((i for i in range(T * k) if flat[i] != -1), key=lambda i: (flat[i], i))
    srt_tok, srt_w, offsets, counts, tiles = [], [], [0], [], []
    pos = [-1] * (T * k)
    for e in range(E):
        mine = [i for i in order if flat[i] == e]
        counts.append(len(mine))
        for i in mine:
            pos[i] = len(srt_tok)
            srt_tok.append(i // k)
            srt_w.append(wf[i])
        while len(srt_tok) % tm:
            srt_tok.append(-1)
            srt_w.append(0.0)
        n_tiles_before = offsets[-1] // tm
        offsets.append(len(srt_tok))
        tiles += [e] * (offsets[-1] // tm - n_tiles_before)
    return dict(R_pad=len(srt_tok), offsets=offsets, counts=counts, srt_tok=srt_tok,
                srt_w=srt_w, pos=pos, tile_expert=tiles)


def assert_plan_equal(p, b):
    assert p["R_pad"] == b["R_pad"]
    assert p["offsets"].tolist() == b["offsets"]
    assert p["counts"].tolist() == b["counts"]
    assert p["srt_tok"].tolist() == b["srt_tok"]
    # routing weights are copied bit for bit
    assert p["srt_w"].view(np.uint32).tolist() == np.asarray(b["srt_w"], np.float32).view(np.uint32).tolist()
    assert p["pos"].ravel().tolist() == b["pos"]
    assert p["tile_expert"].tolist() == b["tile_expert"]


def check_invariants(ids, w, E, tm, p):
    """The plan's invariants: every routed (token, slot) appears exactly once,
    ranks keep token order inside an expert, pad rows are -1 with weight +0,
    counts sum to the routed entries, offsets are tile multiples, and the
    tile table covers each expert's rows."""
    T, k = ids.shape
    flat = ids.ravel()
    routed = flat != -1
    assert int(p["counts"].sum()) == int(routed.sum())
    assert np.all(p["offsets"] % tm == 0)
    assert np.all(np.diff(p["offsets"]) >= 0)
    assert p["offsets"][0] == 0 and p["offsets"][-1] == p["R_pad"]
    pos = p["pos"].ravel()
    assert np.all(pos[~routed] == -1)
    rows = pos[routed]
    assert len(np.unique(rows)) == len(rows)              # each entry once
    assert np.all(p["srt_tok"][rows] == np.nonzero(routed)[0] // k)
    assert np.all(p["srt_w"][rows].view(np.uint32) == w.ravel()[routed].view(np.uint32))
    pad = np.ones(p["R_pad"], bool)
    pad[rows] = False
    assert np.all(p["srt_tok"][pad] == -1)
    assert np.all(p["srt_w"][pad].view(np.uint32) == 0)
    for e in range(E):
        lo, hi = p["offsets"][e], p["offsets"][e + 1]
        c = p["counts"][e]
        assert hi - lo == -(-c // tm) * tm
        assert np.all(flat[np.nonzero(pos >= 0)[0][(pos[pos >= 0] >= lo) & (pos[pos >= 0] < hi)]] == e)
        toks = p["srt_tok"][lo:lo + c]
        assert np.all(np.diff(toks) >= 0)                  # token order kept
        assert np.all(p["srt_tok"][lo + c:hi] == -1)
        assert np.all(p["tile_expert"][lo // tm:hi // tm] == e)
    assert len(p["tile_expert"]) == p["R_pad"] // tm


def read_cases(path):
    cases, cur = [], None
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {}
        elif key == "end":
            cases.append(cur)
            cur = None
        else:
            cur[key] = vals
    return cases


@pytest.mark.parametrize("case", read_cases(os.path.join(GOLDEN, "plan_worked_example.txt")))
def test_plan_hand_worked(case):
    T, k, E, tm = (int(case[n][0]) for n in ("T", "k", "E", "tm"))
    ids = np.array(case["ids"], np.int32).reshape(T, k)
    w = np.array(case["w"], np.float32).reshape(T, k)
    p = oracle.plan(ids, w, E, tm)
    assert p["R_pad"] == int(case["R_pad"][0])
    assert p["offsets"].tolist() == [int(v) for v in case["offsets"]]
    assert p["counts"].tolist() == [int(v) for v in case["counts"]]
    assert p["srt_tok"].tolist() == [int(v) for v in case["srt_tok"]]
    assert p["srt_w"].tolist() == [float(v) for v in case["srt_w"]]
    assert p["pos"].ravel().tolist() == [int(v) for v in case["pos"]]
    assert p["tile_expert"].tolist() == [int(v) for v in case["tile_expert"]]


@pytest.mark.parametrize("seed", range(12))
def test_plan_vs_brute_force_sort(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 9))
    k = int(rng.integers(1, 4))
    E = int(rng.integers(1, 7))
    tm = int(rng.choice([1, 2, 3, 4, 16]))
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)   # -1 = skipped, duplicates allowed
    w = rng.standard_normal((T, k)).astype(np.float32)
    p = oracle.plan(ids, w, E, tm)
    assert_plan_equal(p, brute_plan(ids, w, E, tm))
    check_invariants(ids, w, E, tm, p)


@pytest.mark.parametrize("tm", [1, 2, 3])
def test_plan_every_id_pattern_t2_e3_k2(tm):
    w = np.array([[0.5, -1.25], [3.0, 0.0625]], np.float32)
    for pat in itertools.product(range(-1, 3), repeat=4):
        ids = np.array(pat, np.int32).reshape(2, 2)
        p = oracle.plan(ids, w, 3, tm)
        assert_plan_equal(p, brute_plan(ids, w, 3, tm))


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
def test_plan_invariants_on_workloads(cfg):
    wl = W.workload(cfg)
    inp = W.make_inputs(wl, weights=False)
    p = oracle.plan(inp["ids"], inp["w"], wl.E, wl.tm)
    check_invariants(inp["ids"], inp["w"], wl.E, wl.tm, p)
    assert p["R_pad"] <= oracle.capacity(wl.T, wl.k, wl.E, wl.tm)


def test_plan_degenerate_cases():
    # all tokens on one expert
    ids = np.full((37, 3), 5, np.int32)
    w = np.arange(111, dtype=np.float32).reshape(37, 3)
    p = oracle.plan(ids, w, 8, 16)
    assert p["R_pad"] == 112 and p["counts"].tolist() == [0] * 5 + [111, 0, 0]
    assert p["srt_tok"][:111].tolist() == [i // 3 for i in range(111)]
    # every slot skipped
    p = oracle.plan(np.full((4, 2), -1, np.int32), np.ones((4, 2), np.float32), 3, 16)
    assert p["R_pad"] == 0 and p["pos"].ravel().tolist() == [-1] * 8
    # zero tokens
    p = oracle.plan(np.zeros((0, 2), np.int32), np.zeros((0, 2), np.float32), 3, 16)
    assert p["R_pad"] == 0 and p["offsets"].tolist() == [0, 0, 0, 0]


def test_plan_rejects_bad_ids_and_small_capacity():
    w = np.ones((2, 2), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.array([[0, 3], [1, 2]], np.int32), w, 3, 4)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.array([[0, -2], [1, 2]], np.int32), w, 3, 4)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.array([[0, 1], [1, 2]], np.int32), w, 3, 4, cap=11)
    assert oracle.plan(np.array([[0, 1], [1, 2]], np.int32), w, 3, 4, cap=12)["R_pad"] == 12


def test_capacity_bound_is_tight():
    # k distinct experts per token, each expert with one row: every expert pads tm-1 rows
    T, k, E, tm = 4, 2, 8, 16
    ids = np.arange(8, dtype=np.int32).reshape(T, k)
    p = oracle.plan(ids, np.ones((T, k), np.float32), E, tm)
    assert p["R_pad"] == oracle.capacity(T, k, E, tm) == T * k + E * (tm - 1)


def test_gather_is_row_copy():
    rng = np.random.default_rng(3)
    x = rng.integers(0, 65536, size=(9, 24), dtype=np.uint16)
    srt_tok = np.array([3, -1, 0, 8, 8, -1, 2], np.int32)
    xs = oracle.gather(x, srt_tok)
    want = np.where((srt_tok >= 0)[:, None], x[np.maximum(srt_tok, 0)], 0).astype(np.uint16)
    assert np.array_equal(xs, want)
