"""The layer captured in a CUDA graph and replayed on new inputs equals eager calls.

switch_forward launches only stream-ordered work, and the router's global exchange keeps
its epoch in device memory (advanced by the last CTA of each launch), so a replayed graph
sees a fresh epoch every time.  Three expert counts cover the router's exchange modes:
one 2-CTA cluster per tile (128 experts), one CTA per SM with the slices meeting in global
memory (200 experts), and CTA pairs sharing each W box (1100 experts); the top-2 layer runs
with both choices taken in the router's own pass (128 experts: one cluster per tile; 200 and
1100: the slices meeting in global memory) and, with d = 192 (not a multiple of 128), in a
pass of its own over the router's float32 logits.
Replays alternate between two inputs; every output is compared bit for bit with an eager
call on the same inputs (the same kernels in the same order).
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
FIELDS_TOP2 = FIELDS + ("expert2", "slot2", "keep2", "gate2", "row2")


def _snapshot(y, r, fields):
    return y.clone(), {f: getattr(r, f).clone() for f in fields}


@pytest.mark.parametrize("E,k,d", [(128, 1, 128), (200, 1, 128), (1100, 1, 128), (128, 2, 128), (200, 2, 128),
                                   (1100, 2, 128), (300, 2, 192)])
def test_graph_replay_equals_eager(E, k, d):
    fields = FIELDS_TOP2 if k == 2 else FIELDS
    shape = LayerShape(f"graph-e{E}-top{k}-d{d}", 1, 900, d, 128, E, 1.0)
    a = make_inputs(shape, 3, "cuda", router_bias_std=0.1)
    b = make_inputs(shape, 4, "cuda", router_bias_std=0.1)
    layer = P.make_layer(shape, top_k=k)
    w = (a["Wr"], a["br"], a["W1"], a["b1"], a["W2"], a["b2"])
    ref = []
    for inp in (a, b):  # eager calls (the first one also warms the library's caches)
        y, r = layer.forward(inp["x"], *w)
        torch.cuda.synchronize()
        ref.append(_snapshot(y, r, fields))
    xs = a["x"].clone()
    rs = layer.alloc_route()
    ys = torch.empty_like(xs)
    layer.forward(xs, *w, r=rs, y=ys)  # one more eager call on the graph's buffers
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        layer.forward(xs, *w, r=rs, y=ys)
    for i in (0, 1, 0, 1):
        xs.copy_((a, b)[i]["x"])
        g.replay()
        torch.cuda.synchronize()
        y_ref, r_ref = ref[i]
        assert torch.equal(ys, y_ref), f"replay on input {i}: y differs from the eager call"
        for f in fields:
            assert torch.equal(getattr(rs, f), r_ref[f]), f"replay on input {i}: {f} differs"
    layer.sync_status()
