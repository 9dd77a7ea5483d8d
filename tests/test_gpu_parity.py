"""GPU parity: the CUDA layer (through the C ABI) against the fp64 oracle.

Small shapes span several routing tiles, ragged tails, both FFN paths (tensor
cores and CUDA cores), float32 and bfloat16, exact ties, E = 1, T = 0 and
capacity overrides; the five named workloads run at full size, with routing
compared in full and the FFN / output on sampled tokens.
"""
import dataclasses

import numpy as np
import pytest
import torch

from gen import LayerShape, WORKLOADS, make_inputs, workload_seed
from oracle import switch_oracle as so
import parity as P  # tests/ is on sys.path under pytest's default import mode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def run_stages(shape, inp, resid=False):
    """route, dispatch, expert_ffn, combine as separate C-ABI calls, then forward."""
    layer = P.make_layer(shape, write_probs=True, write_logits=True, debug_bounds=True)
    r = layer.route(inp["x"], inp["Wr"], inp["br"])
    xe = layer.dispatch(inp["x"], r)
    ye = layer.expert_ffn(xe, inp["W1"], inp["b1"], inp["W2"], inp["b2"], r.expert_rows)
    y = layer.combine(ye, r, inp["x"] if resid else None)
    y2, r2 = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                           inp["x"] if resid else None)
    layer.sync_status()
    torch.cuda.synchronize()
    return layer, r, xe, ye, y, y2, r2


SMALL = {
    # tensor-core FFN path (d, d_ff multiples of 128); 3 routing tiles per group, ragged tail
    "tc-ragged": (LayerShape("tc-ragged", 2, 300, 256, 384, 8, 1.0), dict(expert_bias_std=0.05,
                                                                          router_bias_std=0.1)),
    # expert blocks of 313 rows: two 256-row token chunks, the second partly filled (loaded as
    # 64-row boxes, two atoms per stage)
    "tc-long-expert": (LayerShape("tc-long-expert", 1, 1000, 128, 256, 4, 1.25), {}),
    # CUDA-core FFN path for widths the tensor-core tiles do not take
    "simt-bf16": (LayerShape("simt-bf16", 3, 129, 72, 40, 5, 0.8), dict(expert_bias_std=0.05)),
    # the toy shape in float32 with biases
    "fp32-toy": (dataclasses.replace(WORKLOADS["tiny-e16-fp32"], name="fp32-toy", T=200, G=2),
                 dict(expert_bias_std=0.05)),
    # exact logit ties between experts (0,1), (2,3), (4,5)
    "ties": (LayerShape("ties", 2, 256, 128, 128, 6, 1.0), dict(tie_pairs=3)),
    "one-expert": (LayerShape("one-expert", 1, 50, 128, 128, 1, 0.5), {}),
    "override": (LayerShape("override", 1, 64, 128, 128, 4, 1.0, capacity_override=8), {}),
    "capacity-over-T": (LayerShape("capacity-over-T", 2, 64, 128, 128, 4, 8.0), {}),
    "many-experts": (LayerShape("many-experts", 1, 700, 128, 128, 300, 1.0), {}),
    # token tiles of >= 128 rows with d, d_ff multiples of 256: FFN tiles of two 128-row weight
    # blocks sharing the token tile; 150 rows -> one TMEM accumulator set, 128 -> two
    "tc-two-blocks": (LayerShape("tc-two-blocks", 1, 600, 256, 512, 4, 1.0), dict(expert_bias_std=0.05)),
    "tc-two-blocks-db": (LayerShape("tc-two-blocks-db", 1, 512, 256, 512, 4, 1.0), dict(router_bias_std=0.1)),
    # 350-row expert blocks with two weight blocks per tile and uneven loads: experts that fit
    # one 256-row chunk, and second chunks of one or two 64-row boxes
    # d, d_ff multiples of 512: tiles of four weight blocks on CTA pairs (two blocks per CTA,
    # half of each token chunk in each CTA); 150-row blocks, then 350-row blocks in two chunks
    "tc-pairs": (LayerShape("tc-pairs", 1, 600, 512, 1024, 4, 1.0), dict(expert_bias_std=0.05)),
    "tc-pairs-chunks": (LayerShape("tc-pairs-chunks", 2, 700, 512, 1024, 4, 1.0),
                        dict(expert_bias_std=0.05, router_bias_std=0.3)),
    "tc-chunks-256": (LayerShape("tc-chunks-256", 2, 700, 256, 512, 4, 1.0),
                      dict(expert_bias_std=0.05, router_bias_std=0.3)),
    # d = 192: three 64-column atoms, so the router's last two-atom stage has a zero-filled half
    "odd-atoms": (LayerShape("odd-atoms", 2, 260, 192, 256, 12, 1.0), dict(router_bias_std=0.1)),
    # router slices meeting in global memory.  One tile of 300 experts (5 slices of 64)
    "gx-single-tile": (LayerShape("gx-single-tile", 1, 100, 128, 128, 300, 1.0), dict(router_bias_std=0.1)),
    # 200 experts: 4 slices of 64
    "gx-e200": (LayerShape("gx-e200", 1, 900, 128, 128, 200, 1.0), dict(router_bias_std=0.1)),
    # 512 experts: 8 slices of 64 over 34 tiles (272 items, more than one per SM; some tiles'
    # slices straddle two rounds of the grid)
    "gx-rounds": (LayerShape("gx-rounds", 2, 2100, 128, 128, 512, 1.0), dict(router_bias_std=0.1)),
    # an odd number of tiles (5) over 5 slices of 128 experts
    "gx-odd-tiles": (LayerShape("gx-odd-tiles", 1, 600, 128, 128, 640, 1.0), {}),
    # 1536 experts (6 slices of 256) over 42 tiles: CTA pairs, 126 pair items
    "gx-e1536": (LayerShape("gx-e1536", 1, 5300, 128, 128, 1536, 1.0), dict(router_bias_std=0.1)),
    # 1100 experts (5 slices of 256) over 5 tiles: the last pair's second tile is past the end
    "gx-pair-odd": (LayerShape("gx-pair-odd", 1, 600, 128, 128, 1100, 1.0), {}),
    # two routing groups of 5 tiles: the pair (4, 5) takes the last tile of group 0 and the
    # first of group 1
    "gx-pair-groups": (LayerShape("gx-pair-groups", 2, 600, 128, 128, 1100, 1.0), dict(router_bias_std=0.1)),
    # d > 1024 with 256-expert slices: the hi piece in an accumulator of its own (up to
    # d = 1024 all three pieces share one, two tiles' sets in TMEM: the widest such case next)
    "gx-pair-wide": (LayerShape("gx-pair-wide", 1, 400, 1152, 128, 1100, 1.0), dict(router_bias_std=0.1)),
    "gx-pair-1024": (LayerShape("gx-pair-1024", 1, 400, 1024, 128, 1100, 1.0), dict(router_bias_std=0.1)),
    # float32 rows of 49,408 bytes: too wide for the shared-memory row slots of the bulk-copy
    # dispatch and combine, so their register kernels run
    "wide-rows": (LayerShape("wide-rows", 1, 40, 12352, 32, 4, 1.0, dtype="f32"), dict(expert_bias_std=0.05)),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_shapes_against_oracle(name):
    shape, kw = SMALL[name]
    inp = make_inputs(shape, 7, "cuda", **kw)
    layer, r, xe, ye, y, y2, r2 = run_stages(shape, inp)
    ref, subst = P.oracle_route(inp, shape, P.to_np(r.logits))
    P.compare_route(r, ref, shape)
    P.compare_route(r2, ref, shape)
    P.check_dispatch(xe, inp["x"], ref)
    tokens = np.arange(shape.N)
    outs = P.oracle_outputs(inp, ref, tokens)
    P.check_expert_rows(ye, ref, outs)
    P.check_y(y, ref, outs, tokens)
    assert torch.equal(y, y2), "forward differs from the stage-by-stage calls"
    # every logit written for verification is within 1e-5 of the oracle's float64 logit,
    # whether or not the group's choices were taken from the GPU's logits
    P.check_logits(P.to_np(r.logits), ref)


def test_fused_residual():
    shape, kw = SMALL["tc-ragged"]
    inp = make_inputs(shape, 11, "cuda", **kw)
    layer, r, xe, ye, y, y2, r2 = run_stages(shape, inp, resid=True)
    ref, _ = P.oracle_route(inp, shape, P.to_np(r.logits))
    P.compare_route(r, ref, shape)
    tokens = np.arange(shape.N)
    outs = P.oracle_outputs(inp, ref, tokens)
    P.check_y(y, ref, outs, tokens, resid=inp["x"])
    assert torch.equal(y, y2)
    # dropped tokens carry exactly x through
    dropped = torch.as_tensor(np.flatnonzero(~ref.keep), device="cuda")
    assert torch.equal(y[dropped], inp["x"][dropped])


def test_empty_batch():
    shape = LayerShape("empty", 2, 0, 128, 128, 4, 1.0)
    inp = make_inputs(shape, 1, "cuda")
    layer, r, xe, ye, y, y2, r2 = run_stages(shape, inp)
    assert y.numel() == 0
    assert (r.raw_count == 0).all() and (r.accepted_count == 0).all() and (r.expert_rows == 0).all()
    assert (r.P == 0).all() and float(r.aux_loss) == 0.0
    st = layer.get_stats(r)
    assert st["dropped"] == 0 and st["aux_loss"] == 0.0


# ------------------------------------------------------------------ page examples on the GPU

def _layer_for(G, T, d, F, E, c, override=0):
    return P.make_layer(LayerShape("pin", G, T, d, F, E, c, capacity_override=override),
                        write_probs=True, write_logits=True, debug_bounds=True)


def test_uniform_probabilities_overflow(golden):
    g = golden("uniform_probs_overflow.json")
    T, E = g["T"], g["E"]
    layer = _layer_for(1, T, 128, 128, E, g["capacity_factor"])
    x = torch.randn(T, 128, device="cuda").bfloat16()
    Wr = torch.zeros(E, 128, device="cuda")
    r = layer.route(x, Wr)
    st = layer.get_stats(r)
    assert (r.expert == g["expert_all"]).all()
    assert layer.C == g["C"]
    assert st["accepted_count"] == g["accepted"]
    assert st["dropped"] / T == g["overflow_fraction"]
    assert float(r.balance[0]) == pytest.approx(g["balance"], rel=1e-6)
    assert torch.all(r.probs == 0.25)


def test_truncation_and_shift(golden):
    g = golden("truncation_equal_accepted.json")
    raw = g["raw"]
    E, T = len(raw), sum(raw)
    a = np.concatenate([np.full(n, e) for e, n in enumerate(raw)])[np.random.default_rng(1).permutation(T)]
    x = torch.zeros(T, 128)
    x[torch.arange(T), torch.as_tensor(a)] = 1.0
    x = x.bfloat16().cuda()
    Wr = torch.zeros(E, 128, device="cuda")
    Wr[:, :E] = 4.0 * torch.eye(E, device="cuda")
    layer = _layer_for(1, T, 128, 128, E, 1.0, override=g["C"])
    r0 = layer.route(x, Wr)
    st = layer.get_stats(r0)
    assert st["raw_count"] == raw and st["accepted_count"] == g["accepted"]
    p0 = r0.probs.clone()
    e0 = r0.expert.clone()
    # +100 on every logit: probabilities and choices unchanged
    shift = golden("shift_invariance.json")["shift"]
    r1 = layer.route(x, Wr, torch.full((E,), shift, device="cuda"))
    assert torch.equal(r1.expert, e0)
    torch.testing.assert_close(r1.probs, p0, rtol=1e-5, atol=0)


def test_gate_not_renormalised(golden):
    g = golden("gate_not_renormalised.json")
    q = g["p_selected"]
    d = 128
    x = torch.zeros(1, d)
    x[0, 0] = 1.0
    x = x.bfloat16().cuda()
    Wr = torch.zeros(2, d, device="cuda")
    Wr[0, 0] = float(np.log(q / (1 - q)))
    W1 = torch.zeros(2, 128, d)
    W1[0, 0, 0] = 2.0
    W2 = torch.zeros(2, d, 128)
    W2[0, 0, 0] = 3.0
    layer = _layer_for(1, 1, d, 128, 2, 2.0)
    y, r = layer.forward(x, Wr, None, W1.bfloat16().cuda(), None, W2.bfloat16().cuda(), None)
    assert int(r.expert[0]) == 0
    assert float(r.gate[0]) == pytest.approx(g["gate"], rel=1e-6)
    assert float(y[0, 0]) == pytest.approx(g["gate"] * 6.0, rel=1e-2)  # not 6.0


def test_local_overflow(golden):
    g = golden("local_overflow.json")
    T, E, A = g["T"], g["E"], 3
    a = [A] * g["tokens_to_A"] + [e for e in range(E) if e != A] * 8
    a = np.array(a[:T])[np.random.default_rng(3).permutation(T)]
    x = torch.zeros(T, 128)
    x[torch.arange(T), torch.as_tensor(a)] = 1.0
    Wr = torch.zeros(E, 128)
    Wr[:, :E] = 5.0 * torch.eye(E)
    layer = _layer_for(1, T, 128, 128, E, g["capacity_factor"])
    r = layer.route(x.bfloat16().cuda(), Wr.cuda())
    st = layer.get_stats(r)
    assert st["accepted_count"][A] == g["accepted_A"] and st["dropped"] == g["dropped"]


# ------------------------------------------------------------------ the named workloads at full size

@pytest.mark.parametrize("name", list(WORKLOADS))
def test_named_workload_full_size(name):
    shape = WORKLOADS[name]
    inp = make_inputs(shape, workload_seed(name), "cuda")
    layer = P.make_layer(shape, write_probs=True, write_logits=True)
    y, r = layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    layer.sync_status()
    z_gpu = P.to_np(r.logits)
    ref, subst = P.oracle_route(inp, shape, z_gpu)
    # the router GEMM: every logit against the float64 oracle, before any choice is taken
    # from the GPU's logits
    worst = P.check_logits(z_gpu, ref)
    ties = P.near_tie_tokens(z_gpu, ref.logits)
    del z_gpu
    # integers bit-exact; probabilities, gates, P, balance, aux and z-loss against float64
    # for every token (near ties only let the GPU's logits pick the choices)
    P.compare_route(r, ref, shape)
    # y: every token at switch-base; elsewhere a random sample plus the tokens at every expert
    # block's edges (first and last kept row, both sides of each 256-row chunk boundary)
    if name in ("switch-base-e128", "tiny-e16-fp32"):
        tokens = np.arange(shape.N)
    else:
        tokens = np.union1d(P.sample_tokens(ref, 384, seed=5),
                            P.structured_tokens(ref, 256, max_experts=256 if shape.E > 256 else None, seed=5))
    outs = P.oracle_outputs(inp, ref, tokens)
    P.check_y(y, ref, outs, tokens)
    # every dropped token's output is exactly zero
    dropped = torch.as_tensor(np.flatnonzero(~ref.keep), device="cuda")
    if dropped.numel():
        assert (y[dropped] == 0).all()
    print(f"{name}: max |z - z_ref| {worst:.2e}; near-tie tokens {ties}; groups routed from the GPU's logits "
          f"{len(subst)} of {shape.G}; y checked on {tokens.size} tokens ({int(ref.keep[tokens].sum())} kept)")
    del layer
    torch.cuda.empty_cache()
