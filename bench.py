"""Benchmark of the top-1 Switch MoE layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one switch_forward (router, top-1, slots, capacity mask, statistics,
aux loss, dispatch, expert FFN, combine) over one batch of synthetic tokens
already resident in HBM.  The default workload is the largest layer that fits one
GPU: 2048 experts (the Switch-C expert count), d_model 768, d_ff 2048, capacity
factor 1.0, one routing group of 65536 tokens (12.9 GB of expert weights).
--workload picks one of the others.  Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on this host instead (a bounded
sample of the same workload), and prints the same line with "impl": "reference".
Under torchrun every rank processes its own batch (weak scaling: routing groups
are independent); ranks share nothing on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gen import WORKLOADS, expert_weights, make_inputs, workload_seed  # noqa: E402

METRIC = "Switch top-1 MoE layer fwd tokens/s on 1 B300; % TC peak; dispatch HBM GB/s"
DEFAULT_WORKLOAD = "many-experts-e2048"
L2_FLUSH_BYTES = 256 << 20  # > 126 MB L2


# ---------------------------------------------------------------- across ranks
def rank_batch_seed(seed: int, rank: int, world: int) -> int:
    """Seed of a rank's token batch: routing groups are independent, so each rank routes its
    own batch (weak scaling) while the expert weights, drawn from `seed`, are replicated."""
    return seed if world == 1 else seed + 7919 * rank


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time (the job is done when every rank is)."""
    if not dist:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step: int, world: int, steps: int, ms: float) -> float:
    """Whole-job tokens/s: the tokens every rank processed over the slowest rank's time."""
    return tokens_per_step * world * steps / (ms * 1e-3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


# ---------------------------------------------------------------- clocks during the timed region
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(sm)
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- algorithmic work per launch
def algorithmic(shape, expert_rows: np.ndarray, N: int):
    """Bytes / FLOPs each stage must move or do (kept rows only, experts with tokens only)."""
    d, F, E = shape.d_model, shape.d_ff, shape.E
    es = 4 if shape.dtype == "f32" else 2
    K = int(expert_rows.sum())
    used = int((expert_rows > 0).sum())
    w_bytes = 2 * used * F * d * es
    return {
        "kept_rows": K,
        "experts_used": used,
        # route: read x and W_r, write 13 B of per-token records + [E] stats
        "route_bytes": N * d * es + E * d * 4 + N * 13,
        # dispatch: read kept rows, write them to the expert blocks
        "dispatch_bytes": 2 * K * d * es,
        # expert FFN with the combine fused in: weights of the used experts, the dispatched
        # rows in, y rows out (h stays on chip / in L2); all N rows of y are written, the
        # dropped ones by the dispatch pass
        "ffn_bytes": w_bytes + K * d * es + K * d * es,
        "ffn_flops": 4.0 * K * d * F,
        "router_flops": 2.0 * N * d * E,
    }


def traffic_from_profiles(kernel: str):
    """DRAM bytes per launch recorded by an ncu capture (profiles/ncu_traffic.txt), or None
    when the kernel's source file changed since the capture (the counters no longer apply)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        for line in open(path, encoding="utf-8"):
            parts = line.split()
            if not parts or parts[0].startswith("#") or parts[0] != kernel:
                continue
            src = os.path.join(ROOT, "sparse_mixture_experts_slots_b300", "csrc", parts[1])
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            if h != parts[2]:
                return None
            return {"dram_bytes_per_launch": int(parts[3])}
    except Exception:
        return None
    return None


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)
class ExpertCache:
    """float64 copies of the expert weights the oracle sample touches (converted once)."""

    def __init__(self, fetch):
        self.fetch, self.cache = fetch, {}

    def __call__(self, e: int):
        if e not in self.cache:
            W1, W2 = self.fetch(e)
            self.cache[e] = (W1.float().cpu().numpy().astype(np.float64), W2.float().cpu().numpy().astype(np.float64))
        return self.cache[e]


def oracle_sample(shape, x, Wr, br, experts, n_ffn_tokens: int, top_k: int = 1, n_route_tokens: int = 8192):
    """Time the fp64 oracle on a bounded sample of the workload: routing of the first T'
    tokens of every group (T' = min(T, n_route_tokens / G): a layer of the same shape on
    those tokens, the whole batch when it is small) + the expert FFN of a sample of its kept
    tokens (kept (token, choice) requests with top-2), the FFN time scaled to all its kept
    tokens.  x, Wr, br: float64 arrays; experts(e) -> float64 (W1[e], W2[e]).
    Returns (tokens/s, detail)."""
    from oracle import switch_oracle as so
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()
    Ts = max(1, min(shape.T, n_route_tokens // shape.G))
    if Ts < shape.T:  # the first Ts tokens of every group (groups are contiguous in x)
        x = np.ascontiguousarray(x.reshape(shape.G, shape.T, -1)[:, :Ts].reshape(shape.G * Ts, -1))
    Ns = shape.G * Ts
    t0 = time.perf_counter()
    if top_k == 2:
        r = so.route_top2(x, Wr, br, shape.G, Ts, shape.E, shape.capacity_factor)
        req_e = np.concatenate([r.expert[r.keep], r.expert2[r.keep2]])  # kept (token, choice) requests
        req_t = np.concatenate([np.flatnonzero(r.keep), np.flatnonzero(r.keep2)])
        req_g = np.concatenate([r.gate[r.keep], r.gate2[r.keep2]])
    else:
        r = so.route(x, Wr, br, shape.G, Ts, shape.E, shape.capacity_factor)
        req_t = np.flatnonzero(r.keep)
        req_e = r.expert[req_t]
        req_g = r.gate[req_t]
    t_route = time.perf_counter() - t0
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(req_t.size, size=min(n_ffn_tokens, req_t.size), replace=False))
    used = np.unique(req_e[pick])
    W = {int(e): experts(int(e)) for e in used}  # marshalling, outside the timed part
    t0 = time.perf_counter()
    for e in used:
        sel = pick[req_e[pick] == e]
        W1, W2 = W[int(e)]
        o = so.expert_ffn(x[req_t[sel]], W1, None, W2, None)
        _ = req_g[sel, None] * o
    t_ffn = time.perf_counter() - t0
    t_total = t_route + t_ffn * req_t.size / max(1, pick.size)
    what = f"all {shape.N} tokens" if Ts == shape.T else \
        f"the first {Ts} of {shape.T} tokens of each of the {shape.G} group(s) ({Ns} tokens, as a layer of its own)"
    return Ns / t_total, {
        "cores": threads,
        "sample": (f"routing of {what} + expert FFN/combine of {pick.size} of its {req_t.size} kept "
                   f"{'requests' if top_k == 2 else 'tokens'}, FFN time scaled by {req_t.size}/{pick.size}"),
        "t_route_s": t_route, "t_ffn_sample_s": t_ffn}


def dropped_counts(r, N: int) -> dict:
    """Tokens whose choice was dropped: first choices, and with top-2 second choices apart."""
    out = {"dropped": int(N - int(r.accepted_count.sum().item()))}
    if r.accepted2_count is not None:
        out["dropped_second"] = int(N - int(r.accepted2_count.sum().item()))
    return out


def host_f64(inp):
    x = inp["x"].float().cpu().numpy().astype(np.float64)
    Wr = inp["Wr"].float().cpu().numpy().astype(np.float64)
    br = None if inp["br"] is None else inp["br"].float().cpu().numpy().astype(np.float64)
    return x, Wr, br


def run_reference(args, shape):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # the host draws x and the router; expert weights are drawn per expert as the sample
    # needs them (the 2048-expert layer's 12.9 GB are not drawn whole on the host)
    seed = workload_seed(args.workload)
    inp = make_inputs(shape, seed, "cpu", with_experts=False)
    x, Wr, br = host_f64(inp)
    experts = ExpertCache(lambda e: expert_weights(shape, seed, e, "cpu"))
    vals = []
    detail = {}
    for i in range(args.warmup + args.steps):
        v, detail = oracle_sample(shape, x, Wr, br, experts, args.ref_ffn_tokens, args.top_k, args.ref_route_tokens)
        if i >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * shape.N / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(shape, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": detail["cores"], "kind": "oracle",
                         "sample": detail["sample"]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(shape, args):
    return {"workload": shape.name, "G": shape.G, "T": shape.T, "d_model": shape.d_model, "d_ff": shape.d_ff,
            "E": shape.E, "capacity_factor": shape.capacity_factor, "top_k": getattr(args, "top_k", 1),
            "global_batch_tokens": shape.N * args.gpus, "parallelism": f"replicas{args.gpus}",
            "l2": "flushed (256 MB write) before every device-timed step, outside its events; expert "
                  "weights (>= 0.6 GB) exceed L2 anyway",
            "router_weights": "bf16 split prepared once at load (switch_prepare_router); every step runs "
                              "the router GEMM, softmax, top-1, statistics, slots, dispatch, FFN, combine"}



# ---------------------------------------------------------------- training step (--train)
FP32_ALU_TFLOPS = 148 * 128 * 2 * 2.032 / 1e3  # SMs x FP32 lanes x FMA x max SM clock (GHz) -> TFLOP/s


def run_train(args, shape):
    """One step = switch_forward in training mode + switch_backward (fixed dy, w_aux = 1,
    w_z = 1e-3).  With bf16 tensor-core shapes the backward's expert products run on the
    tensor cores (roofline: the bf16 peak); otherwise on CUDA cores (the float32 ALU peak,
    unit counts x clock)."""
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from sparse_mixture_experts_slots_b300 import SwitchMoE
    inp = make_inputs(shape, workload_seed(args.workload), dev)
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    layer = SwitchMoE(shape.G, shape.T, shape.d_model, shape.d_ff, shape.E, shape.capacity_factor, dtype=dt,
                      training=True, device=dev)
    r = layer.alloc_route()
    y = torch.empty(shape.N, shape.d_model, dtype=dt, device=dev)
    dy = (torch.randn(shape.N, shape.d_model, generator=torch.Generator().manual_seed(3)) * 0.5).to(dt).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fw = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    bw = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = None
    for i in range(args.warmup + args.steps):
        flush.fill_(1.0)
        k = i - args.warmup
        if k == 0:
            torch.cuda.synchronize(dev)
            clocks = ClockSampler(dev.index)  # sampled over the timed steps
        if k >= 0:
            fw[k][0].record(stream)
        layer.forward(inp["x"], inp["Wr"], inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"], r=r, y=y,
                      stream=stream)
        if k >= 0:
            bw[k].record(stream)
        layer.backward(inp["x"], inp["Wr"], inp["W1"], inp["W2"], r, dy, 1.0, 1e-3, stream=stream)
        if k >= 0:
            fw[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks is not None else None
    layer.sync_status(stream)
    step_ms = sum(a.elapsed_time(b) for a, b in fw) / args.steps
    fwd_ms = sum(a.elapsed_time(b) for (a, _), b in zip(fw, bw)) / args.steps
    bwd_ms = step_ms - fwd_ms
    K = int(r.expert_rows.sum().item())
    N, E, d, F = shape.N, shape.E, shape.d_model, shape.d_ff
    es = 4 if shape.dtype == "f32" else 2
    used = int((r.expert_rows > 0).sum().item())
    R = layer.block_rows
    bwd_flops = 4 * 2.0 * K * d * F + 2 * 2.0 * N * E * d
    # algorithmic bytes of the backward: the used experts' W1 and W2 read once, their float32
    # weight gradients written once (every expert's, unused ones as zeros), the saved
    # activations xe and h and the incoming dy read once, the float32 dx, dWr and the router
    # logits [N, E] read / written once
    bwd_bytes = (2 * used * d * F * es + 2 * E * d * F * 4 + K * (d + F) * es + N * d * es + N * d * 4
                 + E * d * 4 + N * E * 4)
    tf = bwd_flops / (bwd_ms * 1e-3) / 1e12
    gbs = bwd_bytes / (bwd_ms * 1e-3) / 1e9
    hbm, tc_burst, tc_sust, peak_src = peaks()
    tc_shapes = shape.dtype == "bf16" and d % 128 == 0 and F % 128 == 0
    print(json.dumps({
        "metric": METRIC + " (training step: forward + backward)", "value": N / (step_ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(shape, argparse.Namespace(gpus=1, top_k=1)) | {"mode": "train"},
        "forward_ms": fwd_ms, "backward_ms": bwd_ms, "kept_rows": K, "expert_block_rows": R,
        "roofline": ({"bound": "hbm", "kernel": "switch_backward (whole backward)", "achieved": gbs, "peak": hbm,
                      "unit": "GB/s", "frac": gbs / hbm, "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)",
                      "algorithmic_bytes": bwd_bytes, "traffic": None,
                      "tensor": {"achieved_tflops": tf, "peak_tflops": tc_burst, "frac": tf / tc_burst},
                      "note": f"the backward moves {bwd_bytes / 1e9:.2f} GB (weights in, float32 weight "
                              f"gradients out) for {bwd_flops / 1e12:.2f} TFLOP; all its products run on the "
                              "tensor cores"}
                     if tc_shapes else
                     {"bound": "alu", "kernel": "bgemm_kernel (backward products)", "achieved": tf,
                      "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": tf / FP32_ALU_TFLOPS,
                      "peak_source": "derived: 148 SMs x 128 FP32 lanes x 2 (FMA) x 2.032 GHz",
                      "algorithmic_flops": bwd_flops, "traffic": None}),
        "clocks": clk,
    }), flush=True)
    return 0

# ---------------------------------------------------------------- routing step alone (--stage route)
def run_route(args, shape):
    """One step = switch_route (router GEMM, softmax, top-1, statistics, aux and z-loss, slots
    and capacity mask) over the workload's tokens with W_r prepared once; no expert weights
    are allocated.  Roofline of the router kernel: its three bf16 pieces' MMA FLOPs (2 N d E
    each) at the bf16 tensor peak."""
    if not torch.cuda.is_available() or shape.dtype != "bf16":
        print(json.dumps({"metric": METRIC + " (routing step)", "error": "needs a CUDA device and bf16"}))
        return 1
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from sparse_mixture_experts_slots_b300 import SwitchMoE
    inp = make_inputs(shape, workload_seed(args.workload), dev, with_experts=False)
    layer = SwitchMoE(shape.G, shape.T, shape.d_model, shape.d_ff, shape.E, shape.capacity_factor,
                      dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    layer.prepare_router(inp["Wr"], stream=stream)
    r = layer.alloc_route()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        layer.route(inp["x"], None, inp["br"], out=r, stream=stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(dev.index)
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        layer.route(inp["x"], None, inp["br"], out=r, stream=stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    layer.sync_status(stream)
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    flops = 3 * 2.0 * shape.N * shape.d_model * shape.E  # hi, mid and lo pieces
    hbm, tc_burst, tc_sust, peak_src = peaks()
    tf = flops / (ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": METRIC + " (routing step)", "value": shape.N / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(shape, argparse.Namespace(gpus=1, top_k=1)) | {"mode": "route"},
        "roofline": {"bound": "tensor", "kernel": "router_tc_kernel + split-free route (scan, slots)",
                     "achieved": tf, "peak": tc_burst, "unit": "TFLOP/s", "frac": tf / tc_burst,
                     "peak_source": f"{peak_src} bf16_tflops (cuBLAS bf16 GEMM, burst)",
                     "algorithmic_flops": flops, "traffic": None,
                     "note": "the router multiplies three bf16 pieces of the float32 W_r; the stage also "
                             "runs the cross-tile scan and the slots kernel"},
        "clocks": clk,
    }), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def run_gpu(args, shape):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from sparse_mixture_experts_slots_b300 import SwitchMoE

    seed = workload_seed(args.workload)
    inp = make_inputs(shape, seed, dev)
    if world > 1:  # each rank routes its own batch; the expert weights are replicated
        inp["x"] = make_inputs(shape, rank_batch_seed(seed, rank, world), dev, with_experts=False)["x"]
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    mk = lambda prof: SwitchMoE(shape.G, shape.T, shape.d_model, shape.d_ff, shape.E, shape.capacity_factor,
                                dtype=dt, profile=prof, top_k=args.top_k, device=dev)
    layer = mk(False)
    r = layer.alloc_route()
    y = torch.empty(shape.N, shape.d_model, dtype=dt, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # inference: the router weights are split into their bf16 pieces once, at load time
    prepared = shape.dtype == "bf16"
    if prepared:
        layer.prepare_router(inp["Wr"], stream=stream)
    Wr_step = None if prepared else inp["Wr"]

    def step(lay):
        lay.forward(inp["x"], Wr_step, inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"], r=r, y=y,
                    stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step(layer)
    layer.sync_status(stream)
    torch.cuda.synchronize(dev)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    launches = 0
    clocks = ClockSampler(dev.index)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.fill_(float(i))  # > L2, outside the step's events
        ev[i][0].record(stream)
        step(layer)
        ev[i][1].record(stream)
        launches += layer.last_launch_count()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)
    layer.sync_status(stream)

    # ---------------- per-stage times: a profiled pass of the same workload (CUDA events
    # recorded on this stream between the stages; no programmatic overlap across them)
    prof_layer = mk(True)
    if prepared:
        prof_layer.prepare_router(inp["Wr"], stream=stream)
    n_prof = max(3, min(args.steps, 50))
    stage_sum = np.zeros(5)
    for i in range(args.warmup + n_prof):
        for _ in range(4):  # ~1 GB of writes: the host enqueues the whole step while they run,
            flush.fill_(1.0)  # so no launch latency lands between the stage events
        step(prof_layer)
        st = np.array(prof_layer.stage_ms())
        if i >= args.warmup:
            stage_sum += st
    prof_layer.sync_status(stream)
    stage_avg = stage_sum / n_prof  # ms: route, dispatch, ffn (+combine), ffn2, combine
    del prof_layer

    # ---------------- end to end through the C ABI with host buffers (switch_forward_host):
    # every step copies x in from pinned host memory and y and the aux loss back out; the
    # call's own copy streams let one step's copies overlap the neighbouring steps' layer.
    # Wall clock between two device-wide synchronisations (the copy streams included).
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty(shape.N, shape.d_model, dtype=dt).pin_memory()
    aux_host = torch.empty(1, dtype=torch.float32).pin_memory()
    done = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):  # no L2 flush here: x comes from the host every step
        layer.forward_host(x_host, Wr_step, inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                           y_host=y_host, aux_host=aux_host, r=r, done=done[i % 2], stream=stream)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, dist, dev)

    # ---------------- (--sm-budget R,F) two batches in flight: two handles on two streams,
    # each handle's router capped at R CTAs and its FFN at F, so the router of one batch (bound
    # by the tensor cores) runs beside the FFN of the other (bound by the weights' bytes)
    two = None
    if args.sm_budget:
        rc, fc = (int(v) for v in args.sm_budget.split(","))
        x_b = make_inputs(shape, seed + 7919, dev, with_experts=False)["x"]
        lays = [mk(False), mk(False)]
        rr = [lays[0].alloc_route(), lays[1].alloc_route()]
        yy = [torch.empty_like(y), torch.empty_like(y)]
        sts = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        for lay in lays:
            if prepared:
                lay.prepare_router(inp["Wr"], stream=stream)
            lay.set_sm_budget(rc, fc)
        torch.cuda.synchronize(dev)

        def two_step(i):
            j = i % 2
            lays[j].forward((inp["x"], x_b)[j], Wr_step, inp["br"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                            r=rr[j], y=yy[j], stream=sts[j])

        for i in range(max(args.warmup, 4)):
            two_step(i)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        ta, tb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ta.record(stream)
        for st in sts:
            st.wait_event(ta)
        for i in range(args.steps):
            two_step(i)
        for st in sts:
            ev_end = torch.cuda.Event()
            ev_end.record(st)
            stream.wait_event(ev_end)
        tb.record(stream)
        torch.cuda.synchronize(dev)
        two_ms = max_over_ranks(ta.elapsed_time(tb), dist, dev)
        # the same alternating batches on one stream with no budgets and no L2 flush: the
        # like-for-like single-stream time
        for lay in lays:
            lay.set_sm_budget(0, 0)
        sts = [stream, stream]
        for i in range(4):
            two_step(i)
        torch.cuda.synchronize(dev)
        ta.record(stream)
        for i in range(args.steps):
            two_step(i)
        tb.record(stream)
        torch.cuda.synchronize(dev)
        one_ms = max_over_ranks(ta.elapsed_time(tb), dist, dev)
        for lay in lays:
            lay.sync_status(stream)
        two = {"value": job_throughput(shape.N, world, args.steps, two_ms), "unit": "tokens/s",
               "ms_per_step": two_ms / args.steps, "route_ctas": rc, "ffn_ctas": fc,
               "one_stream_ms_per_step": one_ms / args.steps,
               "how": "two handles on two streams, batches alternating between them (two in flight); "
                      "router and FFN CTA budgets from switch_set_sm_budget; no L2 flush (weights > L2); "
                      "CUDA events around all steps"}
        del lays, rr, yy

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    # ---------------- roofline of the dominant kernel (the expert FFN)
    hbm, tc_burst, tc_sust, peak_src = peaks()
    rows = r.expert_rows.cpu().numpy()
    work = algorithmic(shape, rows, shape.N)
    tc_path = shape.dtype == "bf16" and shape.d_model % 128 == 0 and shape.d_ff % 128 == 0
    ffn_ms = stage_avg[2] + stage_avg[3] + (stage_avg[4] if not tc_path else 0.0)
    kern = "ffn_persistent_kernel" if tc_path else "grouped_linear_simt_kernel"
    achieved = work["ffn_bytes"] / (ffn_ms * 1e-3) / 1e9
    tflops = work["ffn_flops"] / (ffn_ms * 1e-3) / 1e12
    # The binding roof is the one whose floor time is longer: algorithmic bytes at the copy
    # bandwidth, or the kept rows' FLOPs at the bf16 burst rate.
    tensor_bound = tc_path and work["ffn_flops"] / (tc_burst * 1e12) > work["ffn_bytes"] / (hbm * 1e9)
    # the recorded captures are of the top-1 layer; a top-2 run has no matching record
    traffic = traffic_from_profiles(f"{kern}:{shape.name}") if args.top_k == 1 else None
    value = job_throughput(shape.N, world, args.steps, total_ms)
    names = ["route", "dispatch", "ffn", "ffn_layer2", "combine"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if shape.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(shape, argparse.Namespace(gpus=world, top_k=args.top_k)),
        "roofline": ({"bound": "tensor", "kernel": kern, "achieved": tflops, "peak": tc_burst, "unit": "TFLOP/s",
                      "frac": tflops / tc_burst, "peak_source": f"{peak_src} bf16_tflops (cuBLAS bf16 GEMM, burst)",
                      "frac_of_sustained": tflops / tc_sust, "algorithmic_flops_per_launch": work["ffn_flops"]}
                     if tensor_bound else
                     {"bound": "hbm", "kernel": kern, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                      "frac": achieved / hbm, "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"}) | {
                     "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                     "algorithmic_bytes_per_launch": work["ffn_bytes"],
                     "kernel_ms": ffn_ms,
                     "timing": "CUDA events around the kernel on its stream, profiled pass of the same workload"},
        "stages_ms": {n: float(v) for n, v in zip(names, stage_avg)},
        "stage_gbs": {"route": work["route_bytes"] / (stage_avg[0] * 1e-3) / 1e9,
                      "dispatch": work["dispatch_bytes"] / (stage_avg[1] * 1e-3) / 1e9,
                      "ffn": achieved},
        "stage_hbm_frac": {"route": work["route_bytes"] / (stage_avg[0] * 1e-3) / 1e9 / hbm,
                           "dispatch": work["dispatch_bytes"] / (stage_avg[1] * 1e-3) / 1e9 / hbm,
                           "route_dispatch": (work["route_bytes"] + work["dispatch_bytes"])
                           / ((stage_avg[0] + stage_avg[1]) * 1e-3) / 1e9 / hbm,
                           "target": "route + dispatch + combine >= 0.70 of HBM (the combine is the "
                                     "FFN's layer-2 epilogue on the tensor-core path)"},
        "ffn_tc_frac": {"achieved_tflops": tflops, "peak_tflops": tc_burst, "frac": tflops / tc_burst,
                        "frac_of_sustained": tflops / tc_sust,
                        "note": f"kept-row FLOPs 4*K*d*d_ff; {peak_src} bf16 burst (and sustained); "
                                + ("tensor bound" if tensor_bound else "weight-bandwidth bound")},
        "ffn_hbm_frac": achieved / hbm,
        "dispatch_hbm_gbs": float(work["dispatch_bytes"] / (stage_avg[1] * 1e-3) / 1e9),
        "kept_rows": work["kept_rows"],
        **dropped_counts(r, shape.N),
        "e2e": {"value": job_throughput(shape.N, world, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()),
                "d2h_bytes_per_step": int(y_host.numel() * y_host.element_size() + 4),
                "ms_per_step": e2e_ms / args.steps,
                "how": "switch_forward_host per step (pinned host x in; y and aux loss out), consecutive "
                       "steps overlapping copies with the layer; host wall clock between device syncs"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if two is not None:
        line["two_streams"] = two
    if not args.no_cpu_baseline and world == 1:
        x64, Wr64, br64 = host_f64(inp)
        cache = ExpertCache(lambda e: (inp["W1"][e], inp["W2"][e]))
        for _ in range(2):  # one untimed warm-up sample (BLAS threads, page faults), then the timed one
            v, det = oracle_sample(shape, x64, Wr64, br64, cache, args.ref_ffn_tokens, args.top_k,
                                   args.ref_route_tokens)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": det["cores"], "kind": "oracle",
                                "sample": det["sample"]}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--ref-ffn-tokens", type=int, default=256)
    ap.add_argument("--ref-route-tokens", type=int, default=8192,
                    help="tokens the fp64 oracle routes per timed sample (the first ones of each group)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sm-budget", default="",
                    help="R,F: also time two batches in flight on two streams, router CTAs <= R, FFN CTAs <= F")
    ap.add_argument("--train", action="store_true",
                    help="time a training step (forward in training mode + switch_backward)")
    ap.add_argument("--stage", default="layer", choices=["layer", "route"],
                    help="route: time the routing step alone (no expert weights)")
    ap.add_argument("--top-k", type=int, default=1, choices=[1, 2],
                    help="2: the top-2 variant (weights = softmax over the two highest scores)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    shape = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, shape)
    if args.stage == "route":
        return run_route(args, shape)
    if args.train:
        return run_train(args, shape)
    return run_gpu(args, shape)


if __name__ == "__main__":
    sys.exit(main())
