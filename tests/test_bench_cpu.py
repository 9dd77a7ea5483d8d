"""Host-side logic of bench.py on CPU (no GPU).

The N > 1 path as two gloo ranks: each rank routes its own batch while the expert weights
are replicated, the timed region's barrier, the max over ranks and the whole-job
throughput; the reference arm runs on rank 0 only.  And the roofline's algorithmic byte /
FLOP counts against a hand count.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from gen import WORKLOADS, make_inputs, workload_seed
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shape = WORKLOADS["tiny-e16-fp32"]
        seed = workload_seed(shape.name)
        inp = make_inputs(shape, seed, "cpu")
        x = make_inputs(shape, bench.rank_batch_seed(seed, rank, world), "cpu", with_experts=False)["x"]
        # replicated weights, distinct batches
        w_sum = torch.tensor([float(inp["W1"].double().sum())], dtype=torch.float64)
        x_sum = torch.tensor([float(x.double().sum())], dtype=torch.float64)
        ws = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        xs = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(ws, w_sum)
        dist.all_gather(xs, x_sum)
        dist.barrier()
        local_ms = 10.0 + 2.5 * rank
        total = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.job_throughput(shape.N, world, 7, total)
        with open(out_path + f".{rank}", "w") as fh:
            json.dump({"w": [float(t) for t in ws], "x": [float(t) for t in xs], "total": total, "value": value}, fh)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    out = str(tmp_path / "rank")
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(out + f".{r}")) for r in range(world)]
    for r in res:
        assert r["w"][0] == r["w"][1], "expert weights must be the same on every rank"
        assert r["x"][0] != r["x"][1], "each rank routes its own batch"
        assert r["total"] == 12.5, "the slowest rank's time"
        assert abs(r["value"] - 32 * 2 * 7 / 12.5e-3) < 1e-6
    assert res[0] == res[1]


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny-e16-fp32", "--steps",
                        "1", "--warmup", "1", "--gpus", "2"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert p.returncode == 0 and p.stdout.strip() == ""


def test_roofline_arithmetic_matches_the_hand_count():
    # switch-base with every expert used and 7484 kept rows: the FFN streams both weight
    # matrices of 128 experts (2 * 128 * 3072 * 768 * 2 B) and moves each kept row in and out
    # (2 * 7484 * 768 * 2 B); FLOPs 4 K d d_ff
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from gen import WORKLOADS
    shape = WORKLOADS["switch-base-e128"]
    rows = np.full(shape.E, 7484 // shape.E, dtype=np.int64)
    rows[: 7484 - rows.sum()] += 1
    w = bench.algorithmic(shape, rows, shape.N)
    assert w["kept_rows"] == 7484 and w["experts_used"] == 128
    assert w["ffn_bytes"] == 2 * 128 * 3072 * 768 * 2 + 2 * 7484 * 768 * 2 == 1230950400
    assert w["ffn_flops"] == 4.0 * 7484 * 768 * 3072
    assert bench.FP32_ALU_TFLOPS == 148 * 128 * 2 * 2.032 / 1e3


def test_oracle_sample_bounds_its_routing():
    # the timed oracle routes the first T' = n_route_tokens / G tokens of every group as a
    # layer of its own when the batch is larger, and the whole batch otherwise
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from gen import LayerShape, make_inputs
    shape = LayerShape("sample", 2, 300, 16, 8, 4, 1.0, dtype="f32")
    inp = make_inputs(shape, 5, "cpu")
    x, Wr, br = bench.host_f64(inp)
    experts = bench.ExpertCache(lambda e: (inp["W1"][e], inp["W2"][e]))
    v, det = bench.oracle_sample(shape, x, Wr, br, experts, 16, 1, n_route_tokens=200)
    assert v > 0 and "the first 100 of 300 tokens of each of the 2 group(s) (200 tokens" in det["sample"]
    v, det = bench.oracle_sample(shape, x, Wr, br, experts, 16, 1, n_route_tokens=8192)
    assert v > 0 and det["sample"].startswith("routing of all 600 tokens")
    v, det = bench.oracle_sample(shape, x, Wr, br, experts, 16, 2, n_route_tokens=200)
    assert v > 0 and "requests" in det["sample"]
    assert np.isfinite(det["t_route_s"])
