"""Expert parallelism across two ranks on CPU (gloo): the library's shard plan and all-to-all
plumbing (sparse_mixture_experts_slots_b300.ep) carrying the oracle's per-rank compute.

Each rank routes its own routing groups, sends every expert block of its dispatched buffer
to the rank owning that expert (with the valid row counts), packs the received rows per
local expert with the plan's permutation, runs its experts, unpacks and sends the outputs
back, and combines.  The result must equal the fp64 oracle's single-rank layer over both
ranks' groups: routing bit-exact, y within 1e-12.  Also checks the plan's ownership
arithmetic.  No GPU: the CUDA data plane (switch_ep_regroup + NCCL) is checked on one GPU
by tests/test_gpu_ep.py, which emulates the ranks without a collective.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
G, T, D, F, E, CF = 2, 40, 16, 12, 6, 0.8


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _weights(seed=5):
    rng = np.random.default_rng(seed)
    return dict(Wr=rng.standard_normal((E, D)) * 0.5, br=rng.standard_normal(E) * 0.2,
                W1=rng.standard_normal((E, F, D)) * 0.3, b1=rng.standard_normal((E, F)) * 0.1,
                W2=rng.standard_normal((E, D, F)) * 0.3, b2=rng.standard_normal((E, D)) * 0.1)


def _tokens(rank):
    return np.random.default_rng(100 + rank).standard_normal((G * T, D))


def _rank_main(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    from oracle import switch_oracle as so
    from sparse_mixture_experts_slots_b300.ep import ExpertShards, all_to_all_rows
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _weights()
        x = _tokens(rank)
        plan = ExpertShards(E, world)
        e0, El = plan.begin(rank), plan.local(rank)
        # local routing and dispatch (oracle), blocks [E, R, d]
        rt = so.route(x, w["Wr"], w["br"], G, T, E, CF)
        xe = so.dispatch(x, rt, E, G)
        R = xe.shape[1]
        # first all-to-all: counts, then the expert blocks
        counts = all_to_all_rows(torch.as_tensor(rt.expert_rows, dtype=torch.int64),
                                 [plan.local(r) for r in range(world)], [El] * world).view(world, El).numpy()
        recv = all_to_all_rows(torch.as_tensor(xe).reshape(-1, D), plan.send_rows(R), plan.recv_rows(rank, R),
                               row_shape=(D,)).numpy()
        # pack per local expert (the plan's permutation), run the experts, unpack
        idx = plan.packed_index(counts, R)
        off, rows = plan.packed_offsets(counts)
        packed = recv[idx]
        out = np.zeros_like(packed)
        start = 0
        for j in range(El):
            n = int(rows[j])
            if n:
                e = e0 + j
                out[start:start + n] = so.expert_ffn(packed[start:start + n], w["W1"][e], w["b1"][e], w["W2"][e],
                                                     w["b2"][e])
            start += n
        back = np.zeros_like(recv)
        back[idx] = out
        # second all-to-all: this rank's blocks from every owner, in expert order
        ye = all_to_all_rows(torch.as_tensor(back), plan.recv_rows(rank, R), plan.send_rows(R),
                             row_shape=(D,)).numpy().reshape(E, R, D)
        y = np.zeros((G * T, D))
        for t in range(G * T):
            if rt.keep[t]:
                y[t] = rt.gate[t] * ye[rt.expert[t], rt.row[t]]
        with open(out_path + f".{rank}", "w") as fh:
            json.dump({"y": y.tolist(), "expert": rt.expert.tolist(), "slot": rt.slot.tolist(),
                       "keep": rt.keep.astype(int).tolist(), "counts": counts.tolist(),
                       "offsets": off.tolist()}, fh)
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_layer_equals_single_rank(tmp_path):
    world, port = 2, _free_port()
    out = str(tmp_path / "ep")
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    sys.path.insert(0, ROOT)
    from oracle import switch_oracle as so
    w = _weights()
    xs = [_tokens(r) for r in range(world)]
    ref, y_ref, _ = so.forward(np.concatenate(xs), w["Wr"], w["br"], w["W1"], w["b1"], w["W2"], w["b2"],
                               world * G, T, E, CF)
    N = G * T
    for r in range(world):
        res = json.load(open(out + f".{r}"))
        sl = slice(r * N, (r + 1) * N)
        assert res["expert"] == ref.expert[sl].tolist()
        assert res["slot"] == ref.slot[sl].tolist()
        assert res["keep"] == ref.keep[sl].astype(int).tolist()
        np.testing.assert_allclose(np.asarray(res["y"]), y_ref[sl], rtol=1e-12, atol=1e-14)
        # counts received from each source: that source's kept rows of this rank's experts
        lo, hi = (r * E) // world, ((r + 1) * E) // world
        for s in range(world):
            assert res["counts"][s] == ref.accepted[s * G:(s + 1) * G, lo:hi].sum(axis=0).tolist()
    assert (~ref.keep).any()


def test_shard_plan_arithmetic():
    sys.path.insert(0, ROOT)
    from sparse_mixture_experts_slots_b300.ep import ExpertShards
    for E_, W_ in ((8, 2), (7, 3), (2048, 8), (5, 5), (130, 4)):
        p = ExpertShards(E_, W_)
        sizes = [p.local(r) for r in range(W_)]
        assert sum(sizes) == E_ and max(sizes) - min(sizes) <= 1
        for e in range(E_):
            r = p.owner(e)
            assert p.begin(r) <= e < p.begin(r + 1)
    with pytest.raises(ValueError):
        ExpertShards(3, 4)
    counts = np.array([[2, 0, 1], [1, 3, 0]])  # [W=2, El=3]
    off, rows = ExpertShards.packed_offsets(counts)
    assert off.tolist() == [[0, 0, 0], [2, 0, 1]] and rows.tolist() == [3, 3, 1]
    idx = ExpertShards.packed_index(counts, R=4)
    # expert 0: source 0 rows 0,1 then source 1 row 0; expert 1: source 1 rows 0..2; expert 2: source 0 row 0
    assert idx.tolist() == [0, 1, 12, 16, 17, 18, 8]
