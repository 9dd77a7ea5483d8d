"""CTA budgets of the persistent router and FFN (switch_set_sm_budget) leave every output unchanged.

A budget only changes which CTA computes which router item or FFN tile, so every output must
equal the uncapped call's bit for bit.  The shapes cover each router exchange (one 2-CTA
cluster per tile: 128 experts; slices meeting in global memory: 200 experts; 1100 experts,
whose uncapped router runs on CTA pairs sharing the W boxes and whose budgeted one runs as
single CTAs; top-2 in the router's pass) and both FFN tilings (one CTA per SM; CTA pairs of
four weight blocks).  The smallest budgets are raised to what the kernels need (a CTA per
router slice, one FFN pair).  Then two handles with budgets run on two streams at once, as a
caller overlapping two batches would, and each output must equal its own handle's uncapped
result.
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

CASES = [
    (LayerShape("budget-clusters", 1, 1500, 256, 512, 128, 1.0), 1),
    (LayerShape("budget-global", 2, 900, 128, 256, 200, 1.0), 1),
    (LayerShape("budget-pairs", 1, 1300, 128, 128, 1100, 1.0), 1),
    (LayerShape("budget-ffn-pairs", 2, 700, 512, 1024, 4, 1.0), 1),
    (LayerShape("budget-top2", 1, 1500, 256, 512, 200, 1.0), 2),
]
BUDGETS = [(1, 1), (5, 3), (12, 7)]


def _run(layer, inp, stream=None):
    r = layer.alloc_route()
    y = torch.empty_like(inp["x"])
    layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"], r=r, y=y,
                  stream=stream)
    return y, r


def _same(a, b, fields, what):
    ya, ra = a
    yb, rb = b
    assert torch.equal(ya, yb), f"{what}: y differs"
    for f in fields:
        assert torch.equal(getattr(ra, f), getattr(rb, f)), f"{what}: {f} differs"


@pytest.mark.parametrize("shape,k", CASES, ids=[c[0].name for c in CASES])
def test_budget_leaves_outputs_unchanged(shape, k):
    fields = FIELDS_TOP2 if k == 2 else FIELDS
    inp = make_inputs(shape, 31, "cuda", expert_bias_std=0.05, router_bias_std=0.1)
    layer = P.make_layer(shape, top_k=k)
    ref = _run(layer, inp)
    torch.cuda.synchronize()
    for rc, fc in BUDGETS:
        layer.set_sm_budget(rc, fc)
        got = _run(layer, inp)
        torch.cuda.synchronize()
        _same(got, ref, fields, f"budget route {rc}, ffn {fc}")
    layer.set_sm_budget(0, 0)
    _same(_run(layer, inp), ref, fields, "budget cleared")
    layer.sync_status()


def test_two_budgeted_handles_on_two_streams():
    shape = LayerShape("budget-streams", 1, 3000, 256, 512, 200, 1.0)
    inps = [make_inputs(shape, 40 + i, "cuda", router_bias_std=0.1) for i in range(2)]
    layers = [P.make_layer(shape) for _ in range(2)]
    refs = [_run(l, i) for l, i in zip(layers, inps)]
    torch.cuda.synchronize()
    for l in layers:
        l.set_sm_budget(20, 100)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    for rep in range(4):
        for j in range(2):
            with torch.cuda.stream(streams[j]):
                outs[j].append(_run(layers[j], inps[j], stream=streams[j]))
    torch.cuda.synchronize()
    for j in range(2):
        for o in outs[j]:
            _same(o, refs[j], FIELDS, f"handle {j} on its own stream")
        layers[j].sync_status()


def test_negative_budget_is_rejected():
    layer = P.make_layer(LayerShape("budget-bad", 1, 64, 128, 128, 4, 1.0))
    with pytest.raises(Exception):
        layer.set_sm_budget(-1, 0)
    with pytest.raises(Exception):
        layer.set_sm_budget(0, -2)


def test_budgeted_forward_in_a_cuda_graph():
    """A budgeted layer captured in a CUDA graph and replayed equals its eager calls."""
    shape = LayerShape("budget-graph", 1, 1300, 128, 256, 1100, 1.0)
    inp = make_inputs(shape, 52, "cuda", router_bias_std=0.1)
    layer = P.make_layer(shape)
    layer.set_sm_budget(24, 40)
    ref = _run(layer, inp)
    torch.cuda.synchronize()
    rs = layer.alloc_route()
    ys = torch.empty_like(inp["x"])
    w = (inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    layer.forward(inp["x"], *w, r=rs, y=ys)  # warm the library's caches outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        layer.forward(inp["x"], *w, r=rs, y=ys)
    for _ in range(3):
        ys.zero_()
        g.replay()
        torch.cuda.synchronize()
        _same((ys, rs), ref, FIELDS, "graph replay under a budget")
    layer.sync_status()

