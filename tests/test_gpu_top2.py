"""GPU parity of the top-2 variant (SWITCH_FLAG_TOP2) against the fp64 oracle's route_top2.

Both choices, their weights, slots (second choices after the expert's kept first choices),
keep flags, rows, counts and statistics; the dispatched rows of both choices; y = the
weighted pair of expert outputs.  Shapes take both FFN paths, ragged tiles, several groups,
crowded experts (second choices dropped) and the 混合专家 page's 16-expert, 48-wide router.
"""
import dataclasses

import numpy as np
import pytest
import torch

from gen import LayerShape, WORKLOADS, make_inputs, workload_seed
import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


CASES = {
    "top2-tc": (LayerShape("top2-tc", 2, 300, 256, 384, 8, 1.0), dict(expert_bias_std=0.05, router_bias_std=0.1)),
    # the page's demo router: 16 experts over 48 inputs, two chosen (float32, CUDA-core FFN)
    "top2-page-fp32": (dataclasses.replace(WORKLOADS["tiny-e16-fp32"], name="top2-page-fp32", T=200, G=2),
                       dict(expert_bias_std=0.05)),
    # a strong bias on expert 0: many first and second choices dropped
    "top2-crowded": (LayerShape("top2-crowded", 1, 500, 128, 256, 6, 0.5), dict(router_bias_std=0.8)),
    "top2-many-experts": (LayerShape("top2-many-experts", 1, 700, 128, 128, 300, 1.0), {}),
    # two 128-row weight blocks per FFN tile, 256-row token chunks
    "top2-two-blocks": (LayerShape("top2-two-blocks", 1, 600, 256, 512, 4, 1.0), dict(expert_bias_std=0.05)),
    # both choices in the router's pass with two 64-expert slices per cluster (100 experts,
    # the second slice partly padding), two groups with ragged tiles
    "top2-cluster": (LayerShape("top2-cluster", 2, 300, 256, 384, 100, 1.0), dict(router_bias_std=0.2)),
    # both choices in the router's pass with 8 slices meeting in global memory (512 experts),
    # two groups with ragged tiles
    "top2-global": (LayerShape("top2-global", 2, 700, 256, 256, 512, 1.0), dict(router_bias_std=0.2)),
    # the same with 128-expert slices (700 experts: 6 slices, the last partly padding)
    "top2-global-128": (LayerShape("top2-global-128", 1, 900, 256, 256, 700, 1.0), dict(router_bias_std=0.2)),
    # 256-expert slices (1100 experts: 5 slices, the last partly padding): the three weight
    # pieces in one accumulator block (d <= 1024), and with d > 1024 the hi piece apart
    "top2-global-256": (LayerShape("top2-global-256", 2, 700, 256, 256, 1100, 1.0), dict(router_bias_std=0.2)),
    "top2-global-256-wide": (LayerShape("top2-global-256-wide", 1, 400, 1152, 128, 1100, 1.0),
                             dict(router_bias_std=0.2)),
}


def _run(shape, inp, resid=False):
    layer = P.make_layer(shape, top_k=2, write_logits=True, debug_bounds=True)
    r = layer.route(inp["x"], inp["Wr"], inp["br"])
    xe = layer.dispatch(inp["x"], r)
    ye = layer.expert_ffn(xe, inp["W1"], inp["b1"], inp["W2"], inp["b2"], r.expert_rows)
    y = layer.combine(ye, r, inp["x"] if resid else None)
    y2, r2 = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                           inp["x"] if resid else None)
    layer.sync_status()
    torch.cuda.synchronize()
    return layer, r, xe, y, y2, r2


@pytest.mark.parametrize("name", list(CASES))
def test_top2_against_oracle(name):
    shape, kw = CASES[name]
    inp = make_inputs(shape, 7, "cuda", **kw)
    layer, r, xe, y, y2, r2 = _run(shape, inp)
    assert layer.C == P.so.capacity(2 * shape.capacity_factor, shape.T, shape.E)
    ref, subst = P.oracle_route_top2(inp, shape, P.to_np(r.logits))
    P.check_logits(P.to_np(r.logits), ref)
    P.compare_route_top2(r, ref, shape)
    P.compare_route_top2(r2, ref, shape)
    P.check_dispatch_top2(xe, inp["x"], ref)
    P.check_y_top2(y, ref, inp, np.arange(shape.N))
    assert torch.equal(y, y2), "forward differs from the stage-by-stage calls"
    if name == "top2-crowded":
        assert (~ref.keep2).sum() > 0 and (~ref.keep).sum() > 0


def test_top2_residual():
    shape, kw = CASES["top2-tc"]
    inp = make_inputs(shape, 13, "cuda", **kw)
    layer, r, xe, y, y2, r2 = _run(shape, inp, resid=True)
    ref, _ = P.oracle_route_top2(inp, shape, P.to_np(r.logits))
    P.check_y_top2(y, ref, inp, np.arange(shape.N), resid=inp["x"])
    assert torch.equal(y, y2)


def test_top2_switch_base_full_size():
    name = "switch-base-e128"
    shape = WORKLOADS[name]
    inp = make_inputs(shape, workload_seed(name), "cuda")
    layer = P.make_layer(shape, top_k=2, write_logits=True)
    y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    layer.sync_status()
    ref, _ = P.oracle_route_top2(inp, shape, P.to_np(r.logits))
    P.check_logits(P.to_np(r.logits), ref)
    P.compare_route_top2(r, ref, shape)
    tokens = np.sort(np.random.default_rng(1).choice(shape.N, 192, replace=False))
    P.check_y_top2(y, ref, inp, tokens)


@pytest.mark.parametrize("E", [100, 200, 1100])
def test_top2_exact_ties_across_slices(E):
    # Router rows duplicated within one 64-expert slice (5 -> 6) and across slices (3 -> 70
    # -> 140 -> 300 where they exist): identical logits, so both choices follow the
    # lowest-index rule through the column-group and slice merges (100 experts: a 2-CTA
    # cluster; 200: slices of 64 meeting in global memory; 1100: slices of 256, expert 300 in
    # the second).  A shift on expert 3 makes it the usual winner.
    shape = LayerShape(f"top2-ties-e{E}", 2, 300, 128, 128, E, 1.0)
    inp = make_inputs(shape, 21, "cuda")
    Wr = inp["Wr"]
    for dst in (70, 140, 300):
        if dst < E:
            Wr[dst].copy_(Wr[3])
    Wr[6].copy_(Wr[5])
    br = torch.zeros(E, dtype=torch.float32, device="cuda")
    for e in (3, 70, 140, 300):
        if e < E:
            br[e] = 0.5
    inp["br"] = br
    layer, r, xe, y, y2, r2 = _run(shape, inp)
    ref, subst = P.oracle_route_top2(inp, shape, P.to_np(r.logits))
    P.compare_route_top2(r, ref, shape)
    P.check_y_top2(y, ref, inp, np.arange(shape.N))
    e1, e2 = P.to_np(r.expert), P.to_np(r.expert2)
    assert ((e1 == 3) & (e2 == 70)).sum() > 0, "the tie between experts 3 and 70 never decided both choices"
