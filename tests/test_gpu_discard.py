"""The FFN's L2 drop of consumed hidden activations leaves every result unchanged.

Outside training the tensor-core FFN drops a token chunk's h from L2 (no write-back to
DRAM) once the chunk's last layer-2 tile has read it.  It does so by itself only where h
outgrows half of L2 with two accumulator sets per CTA (the 2048-expert workload at full
size); the test-only flag makes it do so for every shape.  A drop before the last read would hand a later tile stale DRAM contents, so
each case runs several calls on different inputs through one handle, flag on and off, and
the outputs must be identical bit for bit (the same kernels and tiles otherwise).  The
cases cover single-CTA tiles with one and two weight blocks, partly filled second chunks,
CTA pairs, several routing groups, the stage-by-stage expert FFN and the fused forward.
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


CASES = {
    "one-block": (LayerShape("discard-one-block", 2, 300, 256, 384, 8, 1.0), dict(router_bias_std=0.1)),
    "long-expert": (LayerShape("discard-long-expert", 1, 1000, 128, 256, 4, 1.25), {}),
    "two-blocks": (LayerShape("discard-two-blocks", 2, 700, 256, 512, 4, 1.0),
                   dict(expert_bias_std=0.05, router_bias_std=0.3)),
    "pairs": (LayerShape("discard-pairs", 2, 700, 512, 1024, 4, 1.0), dict(expert_bias_std=0.05, router_bias_std=0.3)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_discard_leaves_results_unchanged(name):
    shape, kw = CASES[name]
    w = make_inputs(shape, 5, "cuda", **kw)
    args = (w["Wr"], w["br"], w["W1"], w["b1"], w["W2"], w["b2"])
    xs = [make_inputs(shape, seed, "cuda", with_experts=False)["x"] for seed in (31, 32, 33)]
    plain = P.make_layer(shape)
    drop = P.make_layer(shape, test_discard=True)
    for i, x in enumerate(xs):
        y0, r0 = plain.forward(x, *args, x_residual=x if i == 1 else None)
        y1, r1 = drop.forward(x, *args, x_residual=x if i == 1 else None)
        torch.cuda.synchronize()
        assert torch.equal(r0.expert, r1.expert) and torch.equal(r0.slot, r1.slot)
        assert torch.equal(y0, y1), f"{name}: call {i}: y differs with the L2 drop of h"
        # the stage-by-stage expert FFN on the same handles
        xe = plain.dispatch(x, r0)
        ye0 = plain.expert_ffn(xe, w["W1"], w["b1"], w["W2"], w["b2"], r0.expert_rows)
        ye1 = drop.expert_ffn(xe, w["W1"], w["b1"], w["W2"], w["b2"], r1.expert_rows)
        torch.cuda.synchronize()
        for e in range(shape.E):  # rows past an expert's count are unspecified
            n = int(r0.expert_rows[e])
            assert torch.equal(ye0[e, :n], ye1[e, :n]), f"{name}: call {i}: expert {e} rows differ"
    plain.sync_status()
    drop.sync_status()
