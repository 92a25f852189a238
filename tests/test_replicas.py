"""Host logic of the multi-GPU replicas run, on CPU with gloo (world size 2):
every chunk of a long prompt goes to exactly one rank, ranks line up at the
barrier, and the reported time is the slowest rank's."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from moe_prefill_routing_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    r, w, _ = replicas.init_from_env(backend="gloo")
    replicas.barrier(w)
    slowest = replicas.max_over_ranks(10.0 + r, w)
    q.put((r, w, slowest, replicas.chunks_of_rank(8, r, w), replicas.chunk_of_rank(r, w)))
    replicas.finalize(w)


def test_two_rank_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert all(o[2] == 11.0 for o in out)                 # max over ranks
    chunks = sorted(c for o in out for c in o[3])
    assert chunks == list(range(8))                       # each chunk exactly once
    assert [o[4] for o in out] == [0, 1]


def test_single_rank_needs_no_process_group():
    r, w, l = replicas.init_from_env(backend="gloo") if "WORLD_SIZE" not in os.environ else (0, 1, 0)
    assert (r, w) == (0, 1)
    assert replicas.max_over_ranks(3.5, 1) == 3.5
    assert replicas.chunks_of_rank(8, 0, 1) == list(range(8))
