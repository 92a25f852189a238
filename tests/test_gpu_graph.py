"""The layer forward captured once as a CUDA graph and replayed with new
inputs written into the captured buffers: every launch of the library
(one-launch plan, gather, the two GEMMs with their tensor maps, combine;
the 8-bit path's quantization kernels) must replay unchanged, so each
replay equals an eager call on the same inputs bit for bit (the kernels are
deterministic: a fixed unit per CTA, fixed K and slot orders)."""
import pytest
import torch

from moe_prefill_routing_gb300 import binding as B
from moe_prefill_routing_gb300 import workload as W

from helpers import dev, dev16, dev_weights, inputs

pytestmark = pytest.mark.gpu


def _sets(cfg):
    """The workload's inputs, and a second set: token rows reversed and the
    routing redrawn with another seed (same shapes and distribution)."""
    wl = W.workload(cfg)
    inp = inputs(cfg)
    x = dev16(inp["x"])
    ids1, w1 = W.make_routing(wl.T, wl.E, wl.k, wl.routing, seed=1)
    return (x, dev(inp["ids"]), dev(inp["w"])), (x.flip(0).contiguous(), dev(ids1), dev(w1))


def _replays_match(cfg, forward):
    """forward(x, ids, w, y, ws) launches one layer on the current stream."""
    wl = W.workload(cfg)
    a, b = _sets(cfg)
    x, ids, w = (t.clone() for t in a)  # the captured buffers
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.workspace_bytes(wl.T, wl.d, wl.E, wl.k, wl.f, wl.tm), dtype=torch.uint8,
                     device="cuda")
    eager = {}
    for name, (ex, eids, ew) in (("a", a), ("b", b)):
        ye = torch.empty_like(y)
        forward(ex, eids, ew, ye, torch.empty_like(ws))
        eager[name] = ye
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # first calls (attribute and tensor-map setup) outside the capture
        forward(x, ids, w, y, ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        forward(x, ids, w, y, ws)
    for name, (nx, nids, nw) in (("b", b), ("a", a), ("b", b)):
        x.copy_(nx)
        ids.copy_(nids)
        w.copy_(nw)
        y.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), eager[name].view(torch.int16)), name


@pytest.mark.parametrize("cfg", [1, 3])
def test_layer_forward_graph_replay(cfg):
    Wg, Wu, Wd = dev_weights(cfg)
    tm = W.workload(cfg).tm

    def forward(x, ids, w, y, ws):
        B.layer_forward(x, ids, w, Wg, Wu, Wd, tm, y=y, ws=ws)

    _replays_match(cfg, forward)


def test_f8_layer_graph_replay():
    cfg = 3
    Wg, Wu, Wd = dev_weights(cfg)
    q = [B.quantize_e4m3(t, kmajor=True) for t in (Wg, Wu, Wd)]
    tm = W.workload(cfg).tm

    def forward(x, ids, w, y, ws):
        B.layer_forward_e4m3(x, ids, w, q[0], q[1], q[2], tm, y=y, ws=ws, act_e4m3=True)

    _replays_match(cfg, forward)
