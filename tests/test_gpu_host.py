"""switch_forward_host: the layer on host activations, copies on the handle's own streams.

Consecutive calls alternate two staging slots and overlap their copies with each other's
layer; every call must give exactly what switch_forward gives on device buffers (the same
kernels, each output element written once), with and without a completion event, and its
routing must match the fp64 oracle.
"""
import dataclasses

import pytest
import torch

from gen import LayerShape, WORKLOADS, make_inputs
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


CASES = {
    # tensor-core FFN with the combine fused in, ragged routing tiles
    "host-tc": (LayerShape("host-tc", 2, 300, 256, 384, 8, 1.0), dict(expert_bias_std=0.05, router_bias_std=0.1)),
    # x in four copy pieces with a ragged last one (11000 x 768 bf16)
    "host-pieces": (LayerShape("host-pieces", 1, 11000, 768, 256, 8, 1.0), dict(router_bias_std=0.1)),
    # float32 activations: CUDA-core FFN and a separate combine
    "host-fp32": (dataclasses.replace(WORKLOADS["tiny-e16-fp32"], name="host-fp32", T=200, G=2),
                  dict(expert_bias_std=0.05)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_host_matches_device(name):
    shape, kw = CASES[name]
    w = make_inputs(shape, 11, "cuda", **kw)
    xs = [make_inputs(shape, seed, "cuda", with_experts=False)["x"] for seed in (21, 22, 23)]
    layer = P.make_layer(shape, write_logits=True)
    args = (w["Wr"], w["br"], w["W1"], w["b1"], w["W2"], w["b2"])

    ref = []
    for x in xs:
        y, r = layer.forward(x, *args, x_residual=x)
        ref.append((y.cpu(), r.aux_loss.cpu(), r.expert.cpu(), r.slot.cpu()))
    torch.cuda.synchronize()

    x_h = [x.cpu().pin_memory() for x in xs]
    y_h = [torch.full_like(x_h[0], 7.0).pin_memory() for _ in xs]
    a_h = [torch.full((1,), -1.0).pin_memory() for _ in xs]
    done = [torch.cuda.Event() for _ in xs]
    routes = [layer.alloc_route() for _ in xs]
    for i in range(3):  # three calls back to back: slots 0, 1, 0
        layer.forward_host(x_h[i], *args, y_host=y_h[i], aux_host=a_h[i], residual=True, r=routes[i],
                           done=done[i])
    for i in range(3):
        done[i].synchronize()
        assert torch.equal(y_h[i], ref[i][0]), f"{name}: call {i} y differs from switch_forward"
        assert a_h[i].item() == ref[i][1].item(), f"{name}: call {i} aux loss"
        assert torch.equal(routes[i].expert.cpu(), ref[i][2]) and torch.equal(routes[i].slot.cpu(), ref[i][3])

    # without an event the stream itself waits for the copy out
    y4 = torch.zeros_like(x_h[0]).pin_memory()
    a4 = torch.zeros(1).pin_memory()
    layer.forward_host(x_h[1], *args, y_host=y4, aux_host=a4, residual=True)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(y4, ref[1][0]) and a4.item() == ref[1][1].item()
    layer.sync_status()

    # routing of one host call against the oracle
    inp = dict(w, x=xs[2])
    oref, _ = P.oracle_route(inp, shape, P.to_np(routes[2].logits))
    P.compare_route(routes[2], oref, shape)


def test_forward_host_rejects_missing_buffers():
    shape, kw = CASES["host-tc"]
    w = make_inputs(shape, 11, "cuda", **kw)
    layer = P.make_layer(shape)
    from sparse_mixture_experts_slots_b300._lib import SwitchError
    with pytest.raises(SwitchError):
        layer.forward_host(torch.empty(0), w["Wr"], w["br"], w["W1"], w["b1"], w["W2"], w["b2"],
                           y_host=torch.empty(0))
