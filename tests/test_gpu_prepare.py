"""switch_prepare_router: the router weights split once, later calls passing Wr = NULL.

The layer computed with prepared weights must be bit-identical to the layer computed with
Wr passed (the same kernels read the same bf16 pieces), for switch_route and switch_forward;
a NULL Wr without a preparation, or with float32 activations, is rejected on the host; a
call with a non-NULL Wr replaces the prepared split.
"""
import pytest
import torch

from gen import LayerShape, WORKLOADS, make_inputs
import parity as P
from sparse_mixture_experts_slots_b300 import _lib
from sparse_mixture_experts_slots_b300._lib import SwitchError

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _fwd(layer, inp, Wr):
    return layer.forward(inp["x"], Wr, inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])


def test_prepared_router_matches_passed_weights():
    shape = LayerShape("prep", 2, 300, 256, 384, 8, 1.0)
    inp = make_inputs(shape, 4, "cuda", router_bias_std=0.1)
    layer = P.make_layer(shape, write_logits=True)
    with pytest.raises(SwitchError) as err:  # nothing prepared yet
        layer.route(inp["x"], None, inp["br"])
    assert err.value.status == _lib.SWITCH_ERR_INVALID_ARG
    y_ref, r_ref = _fwd(layer, inp, inp["Wr"])
    layer.sync_status()
    y_ref, logits_ref = y_ref.clone(), r_ref.logits.clone()
    other = torch.randn_like(inp["Wr"]) * 0.05
    layer.prepare_router(other)
    y_o, _ = _fwd(layer, inp, None)  # the prepared weights, not the last passed ones
    layer.prepare_router(inp["Wr"])
    y1, r1 = _fwd(layer, inp, None)
    r2 = layer.route(inp["x"], None, inp["br"])
    layer.sync_status()
    assert torch.equal(y1, y_ref) and torch.equal(r1.logits, logits_ref) and torch.equal(r2.logits, logits_ref)
    assert not torch.equal(y_o, y_ref)
    # a non-NULL Wr replaces the prepared split
    _fwd(layer, inp, other)
    y3, _ = _fwd(layer, inp, None)
    layer.sync_status()
    assert torch.equal(y3, y_o)


def test_prepare_needs_bf16():
    shape = WORKLOADS["tiny-e16-fp32"]
    inp = make_inputs(shape, 4, "cuda")
    layer = P.make_layer(shape)
    with pytest.raises(SwitchError) as err:
        layer.prepare_router(inp["Wr"])
    assert err.value.status == _lib.SWITCH_ERR_UNSUPPORTED
    with pytest.raises(SwitchError) as err:
        layer.route(inp["x"], None, None)
    assert err.value.status == _lib.SWITCH_ERR_INVALID_ARG
