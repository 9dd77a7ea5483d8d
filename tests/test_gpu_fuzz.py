"""Seeded random layer shapes against the fp64 oracle (every token, every stage).

The named cases pin particular tiling paths; these draw the shape itself: activation
dtype, widths that do and do not take the tensor-core tiles (d and d_ff multiples of 128
or not, d below one 64-column atom), 1 to 2048 experts (every router exchange mode: one
cluster, CTAs meeting in global memory, CTA pairs above 1024 experts), 1 to 3 routing groups with ragged
token tiles, capacity factors from 0.3 to 2.5 and capacity overrides, biases on and off, the
residual on and off.  Each case runs the stages one by one and fused, and compares routing
bit for bit (near ties as in parity.py), every logit, the dispatched rows, every expert's
ungated rows and every token's output with the oracle.
"""
import numpy as np
import pytest
import torch

from gen import LayerShape, make_inputs
import parity as P

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def draw_case(k: int):
    """Shape and input options of case k (a fixed draw per k)."""
    rs = np.random.RandomState(9100 + k)
    f32 = rs.rand() < 0.15
    if f32:
        d = int(4 * rs.randint(1, 65))      # rows of 16-byte multiples, up to 256
        F = int(4 * rs.randint(1, 65))
    elif rs.rand() < 0.5:                   # tensor-core FFN tiles
        d = int(128 * rs.randint(1, 7))
        F = int(128 * rs.randint(1, 9))
    else:
        d = int(8 * rs.randint(1, 97))      # any 16-byte row, up to 768
        F = int(8 * rs.randint(1, 65))
    E = int(np.clip(np.round(np.exp(rs.uniform(0.0, np.log(2048.0)))), 1, 2048))
    G = int(rs.randint(1, 4))
    T = int(rs.randint(1, max(2, 2100 // G)))
    c = float(np.round(rs.uniform(0.3, 2.5), 2))
    override = int(rs.randint(1, T + 1)) if rs.rand() < 0.15 else 0
    shape = LayerShape(f"fuzz{k}", G, T, d, F, E, c, dtype="f32" if f32 else "bf16", capacity_override=override)
    kw = dict(router_bias_std=float(rs.choice([0.0, 0.1, 0.4])), expert_bias_std=float(rs.choice([0.0, 0.05])))
    resid = bool(rs.rand() < 0.3)
    return shape, kw, resid


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


def test_draws_cover_the_paths():
    """The fixed draws reach each path at least once."""
    shapes = [draw_case(k)[0] for k in range(N_CASES)]
    assert any(s.dtype == "f32" for s in shapes)
    assert any(s.dtype == "bf16" and s.d_model % 128 == 0 and s.d_ff % 128 == 0 for s in shapes)
    assert any(s.dtype == "bf16" and (s.d_model % 128 or s.d_ff % 128) for s in shapes)
    assert any(s.E > 1024 for s in shapes) and any(256 < s.E <= 1024 for s in shapes)
    assert any(s.E <= 16 for s in shapes)
    assert any(s.G > 1 for s in shapes) and any(s.capacity_override for s in shapes)
