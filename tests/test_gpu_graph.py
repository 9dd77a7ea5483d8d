"""The layer captured in a CUDA graph and replayed on new inputs equals eager calls.

switch_forward launches only stream-ordered work, and the router's global exchange keeps
its epoch in device memory (advanced by the last CTA of each launch), so a replayed graph
sees a fresh epoch every time.  Three expert counts cover the router's exchange modes:
one 2-CTA cluster per tile (128 experts), one CTA per SM with the slices meeting in global
memory (200 experts), and CTA pairs sharing each W box (1100 experts).  Replays alternate
between two inputs; every output is compared bit for bit with an eager call on the same
inputs (the same kernels in the same order).
"""
import pytest
import torch

from gen import LayerShape, make_inputs
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


FIELDS = ("expert", "slot", "keep", "gate", "row", "raw_count", "accepted_count", "P", "aux_loss", "expert_rows")


def _snapshot(y, r):
    return y.clone(), {f: getattr(r, f).clone() for f in FIELDS}


@pytest.mark.parametrize("E", [128, 200, 1100])
def test_graph_replay_equals_eager(E):
    shape = LayerShape(f"graph-e{E}", 1, 900, 128, 128, E, 1.0)
    a = make_inputs(shape, 3, "cuda", router_bias_std=0.1)
    b = make_inputs(shape, 4, "cuda", router_bias_std=0.1)
    layer = P.make_layer(shape)
    w = (a["Wr"], a["br"], a["W1"], a["b1"], a["W2"], a["b2"])
    ref = []
    for inp in (a, b):  # eager calls (the first one also warms the library's caches)
        y, r = layer.forward(inp["x"], *w)
        torch.cuda.synchronize()
        ref.append(_snapshot(y, r))
    xs = a["x"].clone()
    rs = layer.alloc_route()
    ys = torch.empty_like(xs)
    layer.forward(xs, *w, r=rs, y=ys)  # one more eager call on the graph's buffers
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        layer.forward(xs, *w, r=rs, y=ys)
    for k in (0, 1, 0, 1):
        xs.copy_((a, b)[k]["x"])
        g.replay()
        torch.cuda.synchronize()
        y_ref, r_ref = ref[k]
        assert torch.equal(ys, y_ref), f"replay on input {k}: y differs from the eager call"
        for f in FIELDS:
            assert torch.equal(getattr(rs, f), r_ref[f]), f"replay on input {k}: {f} differs"
    layer.sync_status()
