"""GPU parity of switch_backward (top-1, SWITCH_FLAG_TRAINING) against the fp64 oracle's
backward: every gradient (dx, dWr, dbr, dW1, db1, dW2, db2) of
L = sum(dy * y) + w_aux * aux_loss + w_z * z_loss, on the same seeded inputs.

Bound: per tensor, ||g - g_ref|| <= tol ||g_ref|| and max |g - g_ref| <= 5 tol max |g_ref|,
tol = 2e-2 with bfloat16 activations (the GPU keeps h and the expert outputs in bfloat16,
relative rounding 2^-9 per element) and 1e-4 in float32.
"""
import dataclasses

import numpy as np
import pytest
import torch

from gen import LayerShape, WORKLOADS, make_inputs
from oracle import switch_oracle as so
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


CASES = {
    "bwd-tc": (LayerShape("bwd-tc", 2, 300, 256, 384, 8, 1.0), dict(expert_bias_std=0.05, router_bias_std=0.1), False),
    "bwd-fp32": (dataclasses.replace(WORKLOADS["tiny-e16-fp32"], name="bwd-fp32", T=200, G=2),
                 dict(expert_bias_std=0.05), False),
    "bwd-dropped-residual": (LayerShape("bwd-dropped", 1, 400, 128, 256, 6, 0.5), dict(router_bias_std=0.5), True),
    # 64 experts and 1024 tokens: the router's products dWr and dx on the tensor cores too
    # (token chunks of 256 rows, dz in bf16 hi/lo pieces)
    "bwd-tc-router": (LayerShape("bwd-tc-router", 2, 512, 256, 384, 64, 1.0), dict(router_bias_std=0.1), False),
}


def _close(name, got, want, tol):
    g = P.to_np(got)
    err = np.linalg.norm(g - want)
    ref = np.linalg.norm(want)
    assert err <= tol * ref + 1e-30, f"{name}: relative L2 {err / max(ref, 1e-30):.3e} > {tol}"
    assert np.max(np.abs(g - want)) <= 5 * tol * np.max(np.abs(want)) + 1e-30, f"{name}: max abs error"


@pytest.mark.parametrize("name", list(CASES))
def test_backward_against_oracle(name):
    shape, kw, residual = CASES[name]
    inp = make_inputs(shape, 5, "cuda", **kw)
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    dy = (torch.randn(shape.N, shape.d_model, generator=torch.Generator().manual_seed(3)) * 0.5).to(dt).cuda()
    layer = P.make_layer(shape, training=True, write_logits=True)
    y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                         inp["x"] if residual else None)
    w_aux, w_z = 0.7, 0.3
    g = layer.backward(inp["x"], inp["Wr"], inp["W1"], inp["W2"], r, dy, w_aux, w_z, residual)
    layer.sync_status()
    torch.cuda.synchronize()
    ref_r, subst = P.oracle_route(inp, shape, P.to_np(r.logits))
    P.compare_route(r, ref_r, shape)
    over = {gi: P.to_np(r.logits)[gi * shape.T:(gi + 1) * shape.T] for gi in subst}
    f = lambda k: None if inp[k] is None else P.to_np(inp[k])
    ref = so.backward(f("x"), f("Wr"), f("br"), f("W1"), f("b1"), f("W2"), f("b2"), shape.G, shape.T, shape.E,
                      shape.capacity_factor, P.to_np(dy), w_aux, w_z, residual=residual,
                      choice_logits=over or None)
    tol = 1e-4 if shape.dtype == "f32" else 2e-2
    for k in ("dx", "dWr", "dbr", "dW1", "db1", "dW2", "db2"):
        _close(k, g[k], ref[k], tol)
    if name == "bwd-dropped-residual":
        assert (~ref["route"].keep).sum() > 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_without_tokens_writes_zero_gradients(dtype):
    # T = 0: no tokens and no expert rows.  Every weight and bias gradient must come out
    # exactly zero (the outputs start as NaN, so an untouched one fails), on the tensor-core
    # path (bf16, widths multiples of 128) and on the CUDA-core path (float32).
    shape = (LayerShape("bwd-empty", 2, 0, 128, 256, 4, 1.0) if dtype == "bf16"
             else LayerShape("bwd-empty-f32", 2, 0, 48, 32, 16, 1.0, dtype="f32"))
    inp = make_inputs(shape, 5, "cuda", expert_bias_std=0.05)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    layer = P.make_layer(shape, training=True)
    y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    E, d, F = shape.E, shape.d_model, shape.d_ff
    nan = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device="cuda")
    out = dict(dx=nan(0, d), dWr=nan(E, d), dbr=nan(E), dW1=nan(E, F, d), db1=nan(E, F), dW2=nan(E, d, F),
               db2=nan(E, d))
    dy = torch.empty(0, d, dtype=dt, device="cuda")
    g = layer.backward(inp["x"], inp["Wr"], inp["W1"], inp["W2"], r, dy, 0.7, 0.3, out=out)
    layer.sync_status()
    torch.cuda.synchronize()
    for k in ("dWr", "dbr", "dW1", "db1", "dW2", "db2"):
        assert torch.equal(g[k], torch.zeros_like(g[k])), f"{k} is not exactly zero"


def test_backward_needs_training_flag():
    shape, kw, _ = CASES["bwd-tc"]
    inp = make_inputs(shape, 5, "cuda", **kw)
    layer = P.make_layer(shape)  # no training flag
    y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    from sparse_mixture_experts_slots_b300._lib import SwitchError
    with pytest.raises(SwitchError):
        layer.backward(inp["x"], inp["Wr"], inp["W1"], inp["W2"], r, inp["x"])
