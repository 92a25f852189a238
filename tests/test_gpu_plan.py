"""GPU routing plan vs the oracle: bit-exact (offsets, counts, srt_tok,
srt_w, pos, tile_expert), with output buffers poisoned first as in "Round 4
Track C: Prefill MoE Plan ...", section 3 (0xDEADBEEF / 777777), so every
value compared was written by the kernels and rows >= R_pad are untouched."""
import numpy as np
import pytest
import torch

import oracle
from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import dev, inputs

pytestmark = pytest.mark.gpu

POISON_I = np.int32(np.uint32(0xDEADBEEF).view(np.int32))
POISON_W = np.float32(777777.0)


def gpu_plan(ids, w, E, tm):
    T, k = ids.shape
    cap = B.capacity(T, k, E, tm)
    d = "cuda"
    out = dict(
        offsets=torch.full((E + 1,), int(POISON_I), dtype=torch.int32, device=d),
        counts=torch.full((E,), int(POISON_I), dtype=torch.int32, device=d),
        srt_tok=torch.full((max(cap, 1),), int(POISON_I), dtype=torch.int32, device=d),
        srt_w=torch.full((max(cap, 1),), float(POISON_W), dtype=torch.float32, device=d),
        pos=torch.full((T, k), int(POISON_I), dtype=torch.int32, device=d),
        tile_expert=torch.full((max(cap // tm, 1),), int(POISON_I), dtype=torch.int32, device=d),
        ws=torch.full((B.plan_workspace_bytes(T, k, E),), 0x5A, dtype=torch.uint8, device=d),
    )
    o = B.plan(dev(ids), dev(w), E, tm, cap=cap, out=out)
    status = B.read_status(o["ws"])
    return {n: o[n].cpu().numpy() for n in
            ("offsets", "counts", "srt_tok", "srt_w", "pos", "tile_expert")}, status


def assert_same_plan(g, ref, tm):
    R = ref["R_pad"]
    assert g["offsets"].tolist() == ref["offsets"].tolist()
    assert g["counts"].tolist() == ref["counts"].tolist()
    assert np.array_equal(g["srt_tok"][:R], ref["srt_tok"])
    assert np.array_equal(g["srt_w"][:R].view(np.uint32), ref["srt_w"].view(np.uint32))
    assert np.array_equal(g["pos"], ref["pos"])
    assert np.array_equal(g["tile_expert"][:R // tm], ref["tile_expert"])
    # nothing past the padded rows / tiles is written
    assert np.all(g["srt_tok"][R:] == POISON_I)
    assert np.all(g["srt_w"][R:] == POISON_W)
    assert np.all(g["tile_expert"][R // tm:] == POISON_I)


def check(ids, w, E, tm):
    g, status = gpu_plan(ids, w, E, tm)
    ref = oracle.plan(ids, w, E, tm)
    assert status == 0
    assert_same_plan(g, ref, tm)
    return ref


@pytest.mark.parametrize("cfg,chunk", [(1, 0), (2, 0), (3, 0), (4, 0), (5, 0), (5, 7)])
def test_plan_workloads(cfg, chunk):
    wl = W.workload(cfg)
    inp = W.make_inputs(wl, chunk=chunk, weights=False)
    check(inp["ids"], inp["w"], wl.E, wl.tm)


@pytest.mark.parametrize("seed", range(10))
def test_plan_page1_shape_seeds(seed):
    ids, w = W.make_routing(2048, 512, 10, "topk_bias", seed=seed)
    check(ids, w, 512, 16)


EDGE = [
    # T, k, E, tm
    (1, 1, 1, 1), (1, 10, 512, 16), (7, 2, 3, 16), (1023, 10, 512, 16), (1024, 10, 512, 16),
    (1025, 10, 512, 16), (300, 8, 31, 32), (300, 8, 33, 64), (777, 2, 1024, 128),
    (513, 1, 2, 16), (64, 8, 4096, 16), (2049, 10, 512, 1), (100, 3, 5, 1024),
    (97, 256, 300, 16),
]


@pytest.mark.parametrize("T,k,E,tm", EDGE)
def test_plan_edges(T, k, E, tm):
    rng = np.random.default_rng(T * 7919 + k * 31 + E)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    w = rng.standard_normal((T, k)).astype(np.float32)
    check(ids, w, E, tm)


@pytest.mark.parametrize("T", [1, 7, 1023, 1025])
@pytest.mark.parametrize("E", [1, 2, 31, 33, 512, 1024])
@pytest.mark.parametrize("k", [1, 2, 8, 10])
@pytest.mark.parametrize("tm", [16, 128])
def test_plan_sweep(T, E, k, tm):
    # every combination of the ragged sizes; ids uniform over the experts
    # (duplicates inside a token allowed), a tenth of the slots skipped
    rng = np.random.default_rng(T * 1_000_003 + E * 1009 + k * 31 + tm)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[rng.random(ids.shape) < 0.1] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    check(ids, w, E, tm)


def test_plan_all_tokens_one_expert():
    ids = np.full((4096, 8), 77, np.int32)
    w = np.random.default_rng(1).random((4096, 8)).astype(np.float32)
    ref = check(ids, w, 128, 16)
    assert ref["counts"][77] == 4096 * 8


def test_plan_many_empty_experts_and_skips():
    rng = np.random.default_rng(2)
    ids = rng.choice([3, 900, 901, 4000], size=(1500, 6)).astype(np.int32)
    ids[rng.random(ids.shape) < 0.3] = -1
    w = rng.standard_normal(ids.shape).astype(np.float32)
    check(ids, w, 4096, 16)


@pytest.mark.parametrize("T,k,E", [(8192, 8, 128), (8193, 8, 128), (4096, 8, 4096), (4097, 8, 4096)])
def test_plan_one_launch_limit(T, k, E):
    # up to 16 x 4096 entries the plan runs as one cluster launch, above it as
    # the multi-kernel plan; both sides of the limit must match the oracle
    ids, w = W.make_routing(T, E, k, "topk", seed=T)
    check(ids, w, E, 16)


def test_plan_large_block_path():
    # T*k = 140002 entries: 35 blocks of 4096, the last one ragged
    ids, w = W.make_routing(70001, 256, 2, "topk", seed=3)
    check(ids, w, 256, 16)


def test_plan_zero_tokens():
    g, status = gpu_plan(np.zeros((0, 4), np.int32), np.zeros((0, 4), np.float32), 9, 16)
    assert status == 0
    assert g["offsets"].tolist() == [0] * 10 and g["counts"].tolist() == [0] * 9


def test_plan_bad_ids_flag_status_and_are_skipped():
    rng = np.random.default_rng(4)
    ids = rng.integers(0, 40, size=(200, 4)).astype(np.int32)
    w = rng.standard_normal(ids.shape).astype(np.float32)
    bad = ids.copy()
    bad[3, 1], bad[150, 0], bad[199, 3] = 40, -5, 1 << 30
    g, status = gpu_plan(bad, w, 40, 16)
    assert status & B.STATUS_BAD_ID
    fixed = np.where((bad < -1) | (bad >= 40), -1, bad).astype(np.int32)
    assert_same_plan(g, oracle.plan(fixed, w, 40, 16), 16)


def test_plan_weights_copied_bitwise():
    # NaN payloads, -0.0, denormals and infinities travel unchanged
    ids = np.array([[0, 1], [1, 0], [0, 0]], np.int32)
    wb = np.array([[0x7FC01234, 0x80000000], [0x00000001, 0x7F800000], [0xFF800000, 0x3F800000]],
                  np.uint32)
    w = wb.view(np.float32)
    g, status = gpu_plan(ids, w, 2, 16)
    ref = oracle.plan(ids, w, 2, 16)
    assert_same_plan(g, ref, 16)


def test_plan_repeatable():
    inp = inputs(2)
    a, _ = gpu_plan(inp["ids"], inp["w"], 512, 16)
    b, _ = gpu_plan(inp["ids"], inp["w"], 512, 16)
    for n in a:
        assert np.array_equal(a[n], b[n])


def test_plan_ten_million_entries_bit_exact():
    # the size of the plan sweep the benchmark times: 10M entries (k = 10,
    # E = 512), multi-kernel plan, against the oracle's counting sort
    T, k, E, tm = 1 << 20, 10, 512, 16
    rng = np.random.default_rng(10)
    ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
    ids[rng.random(ids.shape) < 0.01] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    check(ids, w, E, tm)


@pytest.mark.parametrize("tm", [1, 16, 128, 1024])
def test_plan_multi_kernel_empty_experts_and_tiles(tm):
    # above the one-launch size, with most experts empty (runs of equal
    # offsets for the tile table's search), a few skipped slots and bad ids
    T, k, E = 20000, 4, 700
    rng = np.random.default_rng(tm)
    used = rng.choice(E, size=90, replace=False)
    ids = rng.choice(used, size=(T, k)).astype(np.int32)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = rng.standard_normal(ids.shape).astype(np.float32)
    check(ids, w, E, tm)


@pytest.mark.parametrize("n_entries", [256 * 4096, 256 * 4096 + 100, 512 * 4096])
def test_plan_column_scan_group_boundaries(n_entries):
    # the column scan prefixes block counts inside groups of 256 blocks of
    # 4096 entries and the expert scan adds the groups' totals: exactly one
    # full group, one full group plus a ragged block, two full groups
    # (k = 4; E = 1000 and 2000: the place kernel finds the lanes of one
    # expert from ballots on two and three groups of id bits)
    k = 4
    T = n_entries // k
    for E in (1000, 2000):
        rng = np.random.default_rng(n_entries + E)
        ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
        ids[rng.random(ids.shape) < 0.02] = -1
        w = rng.standard_normal((T, k)).astype(np.float32)
        check(ids, w, E, 16)


@pytest.mark.parametrize("E", [1024, 1025])
@pytest.mark.parametrize("T", [1000, 20000])
def test_plan_walk_switch(E, T):
    # up to 1024 experts the one-launch plan finds the lanes of one expert
    # through per-warp words in shared memory, above that by
    # __match_any_sync; the multi-kernel plan uses the words up to 512
    # experts and ballots on groups of 5 id bits above; T = 1000 runs the
    # one-launch plan, T = 20000 the multi-kernel plan (k = 8)
    rng = np.random.default_rng(E * 7 + T)
    ids = rng.integers(0, E, size=(T, 8), dtype=np.int32)
    ids[:, 0] = E - 1  # the largest id in every token
    ids[rng.random(ids.shape) < 0.05] = -1
    w = rng.standard_normal(ids.shape).astype(np.float32)
    check(ids, w, E, 16)


@pytest.mark.parametrize("T,k,E", [(30001, 3, 700), (12000, 7, 300), (2000, 37, 1500), (300, 255, 512)])
def test_plan_multi_kernel_odd_k(T, k, E):
    # above the one-launch size with k not a power of two: the token index
    # of each row is the flat index divided by k (by a multiply-high); the
    # lanes of one expert come from shared-memory words (E <= 512) or from
    # ballots on two (E <= 1024) or three groups of id bits (E = 1500)
    rng = np.random.default_rng(T + 97 * k)
    ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
    ids[rng.random(ids.shape) < 0.03] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    check(ids, w, E, 16)


@pytest.mark.parametrize("E", [1, 2, 31, 32, 33, 512, 513, 1024, 1025, 4096])
def test_plan_multi_kernel_expert_counts(E):
    # above the one-launch size the place kernel finds the lanes of one
    # expert in a 32-entry step from per-warp words in shared memory (E <=
    # 512) or from one ballot per id bit, combined in groups of 5 bits (one
    # group up to 32 experts, two up to 1024, three above): both sides of
    # each switch, one expert, and the largest expert count (20001 x 4
    # entries, the last block ragged, skipped slots)
    T, k = 20001, 4
    rng = np.random.default_rng(E + 11)
    ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
    ids[rng.random(ids.shape) < 0.03] = -1
    ids[7, :] = E - 1
    w = rng.standard_normal((T, k)).astype(np.float32)
    check(ids, w, E, 16)


def test_plan_multi_kernel_unaligned_buffers():
    # ids, w and pos starting 4 bytes past a 16-byte boundary: the place
    # kernel then copies ids and weights into shared memory 4 bytes at a time
    T, k, E, tm = 30001, 3, 500, 16
    rng = np.random.default_rng(21)
    ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
    ids[rng.random(ids.shape) < 0.02] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    n = T * k
    ids_buf = torch.zeros(n + 4, dtype=torch.int32, device="cuda")
    w_buf = torch.zeros(n + 4, dtype=torch.float32, device="cuda")
    pos_buf = torch.full((n + 4,), int(POISON_I), dtype=torch.int32, device="cuda")
    ids_d = ids_buf[1:n + 1].view(T, k)
    w_d = w_buf[1:n + 1].view(T, k)
    ids_d.copy_(torch.from_numpy(ids))
    w_d.copy_(torch.from_numpy(w))
    pos_d = pos_buf[1:n + 1].view(T, k)
    assert ids_d.data_ptr() % 16 == 4 and pos_d.data_ptr() % 16 == 4
    cap = B.capacity(T, k, E, tm)
    o = B.plan(ids_d, w_d, E, tm, cap=cap, out={"pos": pos_d})
    assert B.read_status(o["ws"]) == 0
    ref = oracle.plan(ids, w, E, tm)
    R = ref["R_pad"]
    assert o["offsets"].cpu().tolist() == ref["offsets"].tolist()
    assert np.array_equal(o["srt_tok"][:R].cpu().numpy(), ref["srt_tok"])
    assert np.array_equal(o["srt_w"][:R].cpu().numpy().view(np.uint32), ref["srt_w"].view(np.uint32))
    assert np.array_equal(pos_d.cpu().numpy(), ref["pos"])
    assert int(pos_buf[0]) == int(POISON_I) and int(pos_buf[n + 1]) == int(POISON_I)
    assert np.array_equal(o["tile_expert"][:R // tm].cpu().numpy(), ref["tile_expert"])


@pytest.mark.parametrize("seed", range(6))
def test_plan_multi_kernel_random_shapes(seed):
    # above the one-launch size with random shapes: expert counts from 1 to
    # 4096, tm from 1 to 256, Zipf-skewed or uniform ids, skipped slots and a
    # few bad ids, T*k from 65K to 700K entries (ragged last block)
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([1, 7, 96, 500, 1024, 1031, 4096]))
    k = int(rng.integers(1, 12))
    T = int(rng.integers(65536 // k + 1, 700000 // k))
    tm = int(rng.choice([1, 16, 48, 256]))
    if seed % 2:
        pop = 1.0 / np.arange(1, E + 1) ** 1.2
        ids = rng.choice(E, size=(T, k), p=pop / pop.sum()).astype(np.int32)
    else:
        ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
    ids[rng.random(ids.shape) < 0.03] = -1
    bad = rng.random(ids.shape) < 1e-5
    ids[bad] = E + 5
    w = rng.standard_normal((T, k)).astype(np.float32)
    g, status = gpu_plan(ids, w, E, tm)
    assert bool(status & B.STATUS_BAD_ID) == bool(bad.any())
    fixed = np.where(ids >= E, -1, ids).astype(np.int32)
    assert_same_plan(g, oracle.plan(fixed, w, E, tm), tm)
