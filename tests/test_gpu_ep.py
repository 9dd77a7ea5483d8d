"""Expert parallelism on one GPU: W ranks emulated in one process, no collective.

Each emulated rank runs the library's stages (ExpertParallelSwitch: routing and dispatch of
its own groups, switch_ep_regroup + the expert FFN of its experts, the combine); the two
all-to-alls are done here with plain tensor copies between the ranks' buffers, so no kernel
waits on another.  The layer must be bit-identical to one handle over all ranks' groups
(same kernels on the same rows), and the regroup kernel must place every row where the
host-side plan's permutation says.
"""
import numpy as np
import pytest
import torch

from gen import LayerShape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("world,E", [(2, 8), (3, 7)])
def test_emulated_ranks_equal_one_handle(world, E):
    from sparse_mixture_experts_slots_b300 import SwitchMoE, _lib
    from sparse_mixture_experts_slots_b300.ep import ExpertParallelSwitch
    G, T, d, F, c = 2, 300, 256, 384, 1.0
    full = LayerShape("ep-full", world * G, T, d, F, E, c)
    inp = make_inputs(full, 9, "cuda", router_bias_std=0.1, expert_bias_std=0.05)
    N = G * T
    xs = [inp["x"][r * N:(r + 1) * N].contiguous() for r in range(world)]
    ranks = [ExpertParallelSwitch(G, T, d, F, E, c, rank=r, world=world) for r in range(world)]
    plan = ranks[0].shards
    R = ranks[0].R
    lo = [plan.begin(r) for r in range(world + 1)]
    W1 = [inp["W1"][lo[r]:lo[r + 1]].contiguous() for r in range(world)]
    b1 = [inp["b1"][lo[r]:lo[r + 1]].contiguous() for r in range(world)]
    W2 = [inp["W2"][lo[r]:lo[r + 1]].contiguous() for r in range(world)]
    b2 = [inp["b2"][lo[r]:lo[r + 1]].contiguous() for r in range(world)]
    staged = [ranks[r].route_and_dispatch(xs[r], inp["Wr"], inp["br"]) for r in range(world)]
    back = []
    for o in range(world):  # the first exchange, as the owner o receives it
        counts = torch.stack([staged[s][2][lo[o]:lo[o + 1]] for s in range(world)]).contiguous()
        recv_x = torch.stack([staged[s][1][lo[o]:lo[o + 1]] for s in range(world)]).contiguous()
        # the regroup kernel against the plan's permutation
        El = lo[o + 1] - lo[o]
        packed = torch.zeros(El, world * R, d, dtype=torch.bfloat16, device="cuda")
        rows = torch.empty(El, dtype=torch.int32, device="cuda")
        _lib.check(ranks[o].lib.switch_ep_regroup(recv_x.data_ptr(), packed.data_ptr(), counts.data_ptr(),
                                                  rows.data_ptr(), world, El, R, d * 2, 0,
                                                  torch.cuda.current_stream().cuda_stream))
        cnt = counts.cpu().numpy()
        idx = torch.as_tensor(plan.packed_index(cnt, R), device="cuda")
        _, prow = plan.packed_offsets(cnt)
        assert rows.cpu().numpy().tolist() == prow.tolist()
        flat_packed = torch.cat([packed[e, :int(prow[e])] for e in range(El)])
        assert torch.equal(flat_packed, recv_x.view(-1, d)[idx])
        back.append(ranks[o].run_experts(counts, recv_x, W1[o], b1[o], W2[o], b2[o]))
    ys = []
    for s in range(world):  # the return exchange: source s collects its blocks in expert order
        ye = torch.cat([back[o][s] for o in range(world)], dim=0).contiguous()
        ys.append(ranks[s].combine(staged[s][0], ye))
    torch.cuda.synchronize()
    ref = SwitchMoE(world * G, T, d, F, E, c, dtype=torch.bfloat16)
    y_ref, r_ref = ref.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"])
    ref.sync_status()
    for s in range(world):
        sl = slice(s * N, (s + 1) * N)
        for f in ("expert", "slot", "keep", "gate"):
            assert torch.equal(getattr(staged[s][0], f), getattr(r_ref, f)[sl]), f
        assert torch.equal(ys[s], y_ref[sl]), f"rank {s}: y differs from the single-handle layer"
    assert int((r_ref.keep == 0).sum()) > 0
