"""Failure detection on the GPU without a GPU fault.

Every wait in the kernels is bounded (about a second of SM clock); when one runs out the
kernel sets the device error word, finishes without hanging, and the host reads
SWITCH_ERR_DEVICE_TIMEOUT.  A test-only flag makes such a wait run out on purpose: one
layer-1 tile of the expert FFN never publishes its stores, so the layer-2 tiles that need
them wait on a count nothing completes.  Non-finite activations make every router logit of
a token non-finite; the router reports SWITCH_ERR_DEVICE_BOUNDS and routes the token to
expert 0, so every index the later stages use stays in range.  After either, the device
still answers and a fresh handle computes the layer against the oracle.
"""
import time

import numpy as np
import pytest
import torch

from gen import LayerShape, make_inputs
import parity as P
from sparse_mixture_experts_slots_b300 import _lib
from sparse_mixture_experts_slots_b300._lib import SwitchError

pytestmark = pytest.mark.gpu

SHAPE = LayerShape("faults", 1, 512, 256, 512, 4, 1.0)


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _inputs():
    inp = make_inputs(SHAPE, 3, "cuda")
    inp["br"] = torch.tensor([0.5, 0.0, 0.0, 0.0], device="cuda")  # expert 0 surely gets tokens
    return inp


def _forward(layer, inp):
    return layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])


def _layer_is_right(inp):
    """A fresh handle on the same device: routing bit-exact, y within the layer tolerance."""
    layer = P.make_layer(SHAPE, write_logits=True)
    y, r = _forward(layer, inp)
    layer.sync_status()
    ref, _ = P.oracle_route(inp, SHAPE, P.to_np(r.logits))
    P.compare_route(r, ref, SHAPE)
    tokens = np.arange(SHAPE.N)
    P.check_y(y, ref, P.oracle_outputs(inp, ref, tokens), tokens)


def test_bounded_wait_runs_out_and_reports_timeout():
    inp = _inputs()
    layer = P.make_layer(SHAPE, test_stall=True)
    t0 = time.perf_counter()
    y, r = _forward(layer, inp)
    with pytest.raises(SwitchError) as err:
        layer.sync_status()
    waited = time.perf_counter() - t0
    assert err.value.status == _lib.SWITCH_ERR_DEVICE_TIMEOUT
    assert int(r.expert_rows[0]) > 0, "expert 0 received no token: nothing waited"
    assert waited < 30.0, f"the stalled call took {waited:.1f} s"
    # the device still answers, and a fresh handle (no stall flag) computes the layer
    torch.cuda.synchronize()
    _layer_is_right(inp)


def test_non_finite_activations_report_bounds_and_stay_in_range():
    inp = _inputs()
    bad = inp["x"].clone()
    bad[5, 17] = float("nan")
    bad[300, 0] = float("inf")
    layer = P.make_layer(SHAPE)
    y, r = layer.forward(bad, inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    with pytest.raises(SwitchError) as err:
        layer.sync_status()
    assert err.value.status == _lib.SWITCH_ERR_DEVICE_BOUNDS
    E, R = SHAPE.E, layer.block_rows
    e = r.expert.cpu().numpy()
    assert ((e >= 0) & (e < E)).all()
    assert e[5] == 0, "a token whose logits are all NaN goes to expert 0"
    row = r.row.cpu().numpy()
    keep = r.keep.cpu().numpy()
    assert ((row >= -1) & (row < R)).all() and set(np.unique(keep)) <= {0, 1}
    assert ((row >= 0) == (keep == 1)).all()
    assert (r.slot.cpu().numpy() >= 0).all()
    assert int(r.expert_rows.sum()) == int(keep.sum())
    # the handle is usable again: the error word was cleared when it was read
    y2, r2 = _forward(layer, inp)
    layer.sync_status()
    _layer_is_right(inp)
