"""Seeded random layer shapes against the fp64 oracle (every token, every stage).

The named cases pin particular tiling paths; these draw the shape itself: activation
dtype, widths that do and do not take the tensor-core tiles (d and d_ff multiples of 128
or not, d below one 64-column atom), 1 to 2048 experts (every router exchange mode: one
cluster, CTAs meeting in global memory, CTA pairs above 1024 experts), 1 to 3 routing groups with ragged
token tiles, capacity factors from 0.3 to 2.5 and capacity overrides, biases on and off, the
residual on and off.  Each case runs the stages one by one and fused, and compares routing
bit for bit (near ties as in parity.py), every logit, the dispatched rows, every expert's
ungated rows and every token's output with the oracle; the fused call then runs again under
a randomly drawn CTA budget (switch_set_sm_budget) and must give the same bits.  Further draws run the top-2 layer
(routing, dispatch and output of both choices) and the training backward (every gradient)
against the oracle on smaller shapes.
"""
import numpy as np
import pytest
import torch

from gen import LayerShape, make_inputs
from oracle import switch_oracle as so
import parity as P

pytestmark = pytest.mark.gpu

N_CASES = 24
N_TOP2 = 12
N_BACKWARD = 10


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def draw_case(k: int, max_tokens: int = 2100, max_experts: int = 2048, max_width: int = 768):
    """Shape and input options of case k (a fixed draw per k and limits)."""
    rs = np.random.RandomState(9100 + k)
    f32 = rs.rand() < 0.15
    if f32:
        d = int(4 * rs.randint(1, 65))      # rows of 16-byte multiples, up to 256
        F = int(4 * rs.randint(1, 65))
    elif rs.rand() < 0.5:                   # tensor-core FFN tiles
        d = int(128 * rs.randint(1, max_width // 128 + 1))
        F = int(128 * rs.randint(1, 9))
    else:
        d = int(8 * rs.randint(1, max_width // 8 + 1))  # any 16-byte row
        F = int(8 * rs.randint(1, 65))
    E = int(np.clip(np.round(np.exp(rs.uniform(0.0, np.log(float(max_experts))))), 1, max_experts))
    G = int(rs.randint(1, 4))
    T = int(rs.randint(1, max(2, max_tokens // G)))
    c = float(np.round(rs.uniform(0.3, 2.5), 2))
    override = int(rs.randint(1, T + 1)) if rs.rand() < 0.15 else 0
    shape = LayerShape(f"fuzz{k}", G, T, d, F, E, c, dtype="f32" if f32 else "bf16", capacity_override=override)
    kw = dict(router_bias_std=float(rs.choice([0.0, 0.1, 0.4])), expert_bias_std=float(rs.choice([0.0, 0.05])))
    resid = bool(rs.rand() < 0.3)
    return shape, kw, resid


ROUTE_FIELDS = ("expert", "slot", "keep", "gate", "row", "raw_count", "accepted_count", "P", "aux_loss",
                "expert_rows", "logits")


def _same_under_budget(layer, k, args, y_ref, r_ref, fields):
    """The fused forward again under a CTA budget drawn for case k: bit-identical results."""
    rs = np.random.RandomState(9300 + k)
    rc, fc = int(rs.randint(1, 41)), int(rs.randint(1, 41))
    layer.set_sm_budget(rc, fc)
    y3, r3 = layer.forward(*args)
    layer.sync_status()
    torch.cuda.synchronize()
    layer.set_sm_budget(0, 0)
    assert torch.equal(y3, y_ref), f"budget ({rc}, {fc}): y differs"
    for f in fields:
        assert torch.equal(getattr(r3, f), getattr(r_ref, f)), f"budget ({rc}, {fc}): {f} differs"


@pytest.mark.parametrize("k", range(N_CASES))
def test_random_shape_against_oracle(k):
    shape, kw, resid = draw_case(k)
    inp = make_inputs(shape, 40 + k, "cuda", **kw)
    layer = P.make_layer(shape, write_probs=True, write_logits=True, debug_bounds=True)
    x = inp["x"]
    w = (inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    r = layer.route(x, inp["Wr"], inp["br"])
    xe = layer.dispatch(x, r)
    ye = layer.expert_ffn(xe, *w, r.expert_rows)
    y = layer.combine(ye, r, x if resid else None)
    y2, r2 = layer.forward(x, inp["Wr"], inp["br"], *w, x if resid else None)
    layer.sync_status()
    torch.cuda.synchronize()

    ref, _ = P.oracle_route(inp, shape, P.to_np(r.logits))
    P.check_logits(P.to_np(r.logits), ref, f"{shape}: logits")
    P.compare_route(r, ref, shape)
    P.compare_route(r2, ref, shape)
    P.check_dispatch(xe, x, ref)
    tokens = np.arange(shape.N)
    outs = P.oracle_outputs(inp, ref, tokens)
    P.check_expert_rows(ye, ref, outs)
    P.check_y(y, ref, outs, tokens, resid=x if resid else None)
    assert torch.equal(y, y2), f"{shape}: forward differs from the stage-by-stage calls"
    _same_under_budget(layer, k, (x, inp["Wr"], inp["br"], *w, x if resid else None), y2, r2, ROUTE_FIELDS)


def test_draws_cover_the_paths():
    """The fixed draws reach each path at least once."""
    shapes = [draw_case(k)[0] for k in range(N_CASES)]
    assert any(s.dtype == "f32" for s in shapes)
    assert any(s.dtype == "bf16" and s.d_model % 128 == 0 and s.d_ff % 128 == 0 for s in shapes)
    assert any(s.dtype == "bf16" and (s.d_model % 128 or s.d_ff % 128) for s in shapes)
    assert any(s.E > 1024 for s in shapes) and any(256 < s.E <= 1024 for s in shapes)
    assert any(s.E <= 16 for s in shapes)
    assert any(s.G > 1 for s in shapes) and any(s.capacity_override for s in shapes)


@pytest.mark.parametrize("k", range(N_TOP2))
def test_random_shape_top2_against_oracle(k):
    shape, kw, resid = draw_case(100 + k, max_tokens=1500, max_experts=600)
    if shape.E < 2:  # two choices need two experts: the configuration is refused
        from sparse_mixture_experts_slots_b300._lib import SwitchError
        with pytest.raises(SwitchError):
            P.make_layer(shape, top_k=2)
        return
    inp = make_inputs(shape, 60 + k, "cuda", **kw)
    layer = P.make_layer(shape, top_k=2, write_logits=True, debug_bounds=True)
    x = inp["x"]
    w = (inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    r = layer.route(x, inp["Wr"], inp["br"])
    xe = layer.dispatch(x, r)
    ye = layer.expert_ffn(xe, *w, r.expert_rows)
    y = layer.combine(ye, r, x if resid else None)
    y2, r2 = layer.forward(x, inp["Wr"], inp["br"], *w, x if resid else None)
    layer.sync_status()
    torch.cuda.synchronize()
    ref, _ = P.oracle_route_top2(inp, shape, P.to_np(r.logits))
    P.check_logits(P.to_np(r.logits), ref, f"{shape}: logits")
    P.compare_route_top2(r, ref, shape)
    P.compare_route_top2(r2, ref, shape)
    P.check_dispatch_top2(xe, x, ref)
    P.check_y_top2(y, ref, inp, np.arange(shape.N), resid=x if resid else None)
    assert torch.equal(y, y2), f"{shape}: forward differs from the stage-by-stage calls"
    _same_under_budget(layer, 100 + k, (x, inp["Wr"], inp["br"], *w, x if resid else None), y2, r2,
                       ROUTE_FIELDS + ("expert2", "slot2", "keep2", "gate2", "row2"))


@pytest.mark.parametrize("k", range(N_BACKWARD))
def test_random_shape_backward_against_oracle(k):
    shape, kw, resid = draw_case(200 + k, max_tokens=800, max_experts=300, max_width=384)
    inp = make_inputs(shape, 80 + k, "cuda", **kw)
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    dy = (torch.randn(shape.N, shape.d_model, generator=torch.Generator().manual_seed(k)) * 0.5).to(dt).cuda()
    layer = P.make_layer(shape, training=True, write_logits=True)
    y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                         inp["x"] if resid else None)
    w_aux, w_z = 0.7, 0.3
    g = layer.backward(inp["x"], inp["Wr"], inp["W1"], inp["W2"], r, dy, w_aux, w_z, resid)
    layer.sync_status()
    torch.cuda.synchronize()
    _, subst = P.oracle_route(inp, shape, P.to_np(r.logits))
    over = {gi: P.to_np(r.logits)[gi * shape.T:(gi + 1) * shape.T] for gi in subst}
    f = lambda key: None if inp[key] is None else P.to_np(inp[key])
    ref = so.backward(f("x"), f("Wr"), f("br"), f("W1"), f("b1"), f("W2"), f("b2"), shape.G, shape.T, shape.E,
                      shape.capacity_factor, P.to_np(dy), w_aux, w_z, residual=resid, choice_logits=over or None,
                      capacity_override=shape.capacity_override)
    tol = 1e-4 if shape.dtype == "f32" else 2e-2
    for key in ("dx", "dWr", "dbr", "dW1", "db1", "dW2", "db2"):
        got = P.to_np(g[key])
        want = ref[key]
        err = np.linalg.norm(got - want)
        assert err <= tol * np.linalg.norm(want) + 1e-30, f"{shape}: {key} relative L2 {err:.3e}"
        assert np.max(np.abs(got - want)) <= 5 * tol * np.max(np.abs(want)) + 1e-30, f"{shape}: {key} max abs error"
