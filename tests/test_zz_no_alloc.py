"""moe_plan_noalloc, the plan entry point that allocates nothing, against
moe_plan through the C ABI.

It exists for callers that cannot allocate device memory (a serving process
whose memory manager already owns all of the GPU's memory, a plug-in given
buffers by its host application); it keeps the plan's scratch in a fixed
array inside the library.  Its results must equal moe_plan's bit for bit, the
bar every plan test here uses, on two calls in a row, so that whatever the
first call leaves in the shared array cannot leak into the second.  This file
is collected last."""
import numpy as np
import pytest
import torch

import oracle

from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

pytestmark = pytest.mark.gpu

FIELDS = ("offsets", "counts", "srt_tok", "srt_w", "pos", "tile_expert")
MAX_COUNTS = 266240  # MOE_PLAN_NOALLOC_MAX_COUNTS


def _poisoned(T, k, E, cap, tm):
    d = "cuda"
    return dict(offsets=torch.full((E + 1,), -99, dtype=torch.int32, device=d),
                counts=torch.full((E,), -99, dtype=torch.int32, device=d),
                srt_tok=torch.full((cap,), -99, dtype=torch.int32, device=d),
                srt_w=torch.full((cap,), 777777.0, dtype=torch.float32, device=d),
                pos=torch.full((T, k), -99, dtype=torch.int32, device=d),
                tile_expert=torch.full((max(cap // tm, 1),), -99, dtype=torch.int32, device=d))


def _compare(ids_np, w_np, E, tm, with_status=True, against_oracle=False):
    T, k = ids_np.shape
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    cap = B.capacity(T, k, E, tm)
    ref = B.plan(ids, w, E, tm, cap=cap, out=_poisoned(T, k, E, cap, tm))
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda") if with_status else None
    got = B.plan_noalloc(ids, w, E, tm, cap=cap, out=_poisoned(T, k, E, cap, tm), status=status)
    torch.cuda.synchronize()
    R = int(ref["offsets"][E].item())
    for n in FIELDS:
        a, b = ref[n], got[n]
        if n in ("srt_tok", "srt_w"):
            a, b = a[:R], b[:R]
        elif n == "tile_expert":
            a, b = a[:R // tm], b[:R // tm]
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), n
    assert B.read_status(ref["ws"]) == 0
    if with_status:
        assert int(status.item()) == 0
    if against_oracle:
        o = oracle.plan(ids_np, w_np, E, tm)
        Ro = o["R_pad"]
        assert Ro == R
        assert got["offsets"].cpu().numpy().tolist() == o["offsets"].tolist()
        assert got["counts"].cpu().numpy().tolist() == o["counts"].tolist()
        assert np.array_equal(got["srt_tok"][:R].cpu().numpy(), o["srt_tok"])
        assert np.array_equal(got["srt_w"][:R].cpu().numpy().view(np.uint32),
                              o["srt_w"].view(np.uint32))
        assert np.array_equal(got["pos"].cpu().numpy(), o["pos"])
        assert np.array_equal(got["tile_expert"][:R // tm].cpu().numpy(), o["tile_expert"])


def _uniform(T, k, E, seed, skip=0.01):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k), dtype=np.int32)
    ids[rng.random(ids.shape) < skip] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    return ids, w


def test_noalloc_plan_equals_moe_plan_two_calls_in_a_row():
    # call 1: the page-1 plan shape; call 2: another shape with skipped slots
    ids, w = W.make_routing(2048, 512, 10, "topk_bias", seed=0)
    _compare(ids, w, 512, 16)
    rng = np.random.default_rng(5)
    ids2 = rng.integers(0, 300, size=(777, 8)).astype(np.int32)
    ids2[rng.random(ids2.shape) < 0.2] = -1
    w2 = rng.standard_normal(ids2.shape).astype(np.float32)
    _compare(ids2, w2, 300, 32)


def test_noalloc_multi_kernel_path_uses_the_scratch_array():
    # above 64K entries the plan runs as four kernels whose per-block and
    # per-group expert counts live in the library's scratch array: about 1M
    # entries, then the largest size the array takes at E = 512 (2.1M
    # entries: 517 blocks + 3 groups = 520 rows of 512 counts, all of
    # MOE_PLAN_NOALLOC_MAX_COUNTS), then a smaller call
    # with another expert count and fewer blocks, so that whatever a larger
    # call left in the array is there when the smaller one runs; each is
    # compared with moe_plan and with the oracle
    ids, w = _uniform(104858, 10, 512, seed=31)
    _compare(ids, w, 512, 16, against_oracle=True)
    ids, w = _uniform(211763, 10, 512, seed=32)
    blocks = -(-ids.size // 4096)
    assert blocks == 517 and (blocks + -(-blocks // 256)) * 512 == MAX_COUNTS
    _compare(ids, w, 512, 16, against_oracle=True)
    ids, w = _uniform(20001, 4, 300, seed=33, skip=0.05)
    _compare(ids, w, 300, 32, against_oracle=True)


def test_noalloc_without_a_status_word():
    # status = NULL: the call's status bits go to the library's own header
    # word (not readable by the caller); the outputs are unchanged, on both
    # the one-launch and the multi-kernel path
    ids, w = W.make_routing(2048, 512, 10, "topk_bias", seed=3)
    _compare(ids, w, 512, 16, with_status=False)
    ids, w = _uniform(30000, 4, 128, seed=34)
    _compare(ids, w, 128, 16, with_status=False, against_oracle=True)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 74 blocks of 4096 entries x 4096 experts is above MOE_PLAN_NOALLOC_MAX_COUNTS
    T, k, E, tm = 30000, 10, 4096, 16
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.plan_noalloc(ids, w, E, tm)
    assert e.value.code == B.MOE_ERR_WORKSPACE
