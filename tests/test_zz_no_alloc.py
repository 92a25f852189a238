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

from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

pytestmark = pytest.mark.gpu

FIELDS = ("offsets", "counts", "srt_tok", "srt_w", "pos", "tile_expert")


def _poisoned(T, k, E, cap, tm):
    d = "cuda"
    return dict(offsets=torch.full((E + 1,), -99, dtype=torch.int32, device=d),
                counts=torch.full((E,), -99, dtype=torch.int32, device=d),
                srt_tok=torch.full((cap,), -99, dtype=torch.int32, device=d),
                srt_w=torch.full((cap,), 777777.0, dtype=torch.float32, device=d),
                pos=torch.full((T, k), -99, dtype=torch.int32, device=d),
                tile_expert=torch.full((max(cap // tm, 1),), -99, dtype=torch.int32, device=d))


def _compare(ids_np, w_np, E, tm):
    T, k = ids_np.shape
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np).cuda()
    cap = B.capacity(T, k, E, tm)
    ref = B.plan(ids, w, E, tm, cap=cap, out=_poisoned(T, k, E, cap, tm))
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
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
    assert int(status.item()) == B.read_status(ref["ws"]) == 0


def test_noalloc_plan_equals_moe_plan_two_calls_in_a_row():
    # call 1: the page-1 plan shape; call 2: another shape with skipped slots
    ids, w = W.make_routing(2048, 512, 10, "topk_bias", seed=0)
    _compare(ids, w, 512, 16)
    rng = np.random.default_rng(5)
    ids2 = rng.integers(0, 300, size=(777, 8)).astype(np.int32)
    ids2[rng.random(ids2.shape) < 0.2] = -1
    w2 = rng.standard_normal(ids2.shape).astype(np.float32)
    _compare(ids2, w2, 300, 32)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 74 blocks of 4096 entries x 4096 experts is above MOE_PLAN_NOALLOC_MAX_COUNTS
    T, k, E, tm = 30000, 10, 4096, 16
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoeError) as e:
        B.plan_noalloc(ids, w, E, tm)
    assert e.value.code == B.MOE_ERR_WORKSPACE
