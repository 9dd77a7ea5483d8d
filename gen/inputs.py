"""Seeded synthetic inputs for the top-1 Switch MoE layer forward pass.

This module only draws tensors.  It holds none of the layer's arithmetic (no
routing, no softmax, no capacity rule, no FFN), so the fp64 oracle and the CUDA
path can both be fed from it without sharing any of the method.

Workload shapes follow the pages' settings:
  * the 48 -> 32 -> 48 ReLU expert and 16-expert router of the toy model on the
    "混合专家" page (world.lapla.si/zh/moe, section "专家里面是什么");
  * Switch-Base / Switch-Large expert widths and 128 experts (Switch Transformers
    paper card on ai-papers.xuzou.cn, section "证据", Table 1);
  * 2048 experts as in Switch-C (same card, section "证据", Table 9).
Initialisation: the 0.1x init scale of the "按敏感组件设置精度、容量与初始化"
section of the wq-win "Switch Transformer：每个词只选一个专家" page, i.e. a
truncated normal with std sqrt(0.1 / fan_in), redrawn outside +-2 std.

There is no dataset: x ~ N(0, 1) stands in for token representations.  All
draws come from torch's seeded generator on the requested device; a test that
needs the same tensor on the host copies the generated tensor, so both sides
always see identical values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One routing workload: G groups of T tokens, d -> d_ff -> d experts."""

    name: str
    G: int
    T: int
    d_model: int
    d_ff: int
    E: int
    capacity_factor: float
    dtype: str = "bf16"          # activations and expert weights: "bf16" or "f32"
    router_init: str = "normal"  # "normal": N(0, 0.1/d); "trunc": truncated normal
    router_bias: str = "none"    # "none" or "skewed" (see skewed_router_bias)
    bias_gamma: float = 0.0      # scale of the skewed router bias
    capacity_override: int = 0   # >0: use this capacity instead of ceil(cT/E)

    @property
    def N(self) -> int:
        return self.G * self.T


# Calibrated so the skewed-load workload overflows ~25% of its tokens
# (the workload asks for 15-40%); see skewed_router_bias.
SKEW_GAMMA = 0.075

WORKLOADS = {
    "tiny-e16-fp32": LayerShape("tiny-e16-fp32", 1, 32, 48, 32, 16, 1.0,
                                dtype="f32", router_init="trunc"),
    "switch-base-e128": LayerShape("switch-base-e128", 1, 8192, 768, 3072, 128, 1.0),
    "skewed-e64-g8": LayerShape("skewed-e64-g8", 8, 4096, 768, 3072, 64, 1.25,
                                router_bias="skewed", bias_gamma=SKEW_GAMMA),
    "switch-large-e128": LayerShape("switch-large-e128", 1, 32768, 1024, 4096, 128, 1.25),
    "many-experts-e2048": LayerShape("many-experts-e2048", 1, 65536, 768, 2048, 2048, 1.0),
}
WORKLOAD_ORDER = list(WORKLOADS)
# seed = 1000 + the workload's position (1-based) in WORKLOAD_ORDER
WORKLOAD_SEEDS = {name: 1000 + i + 1 for i, name in enumerate(WORKLOAD_ORDER)}

_CHUNK_ELEMS = 1 << 26  # fixed draw chunk, so values never depend on free memory


def act_dtype(shape: LayerShape) -> torch.dtype:
    return torch.float32 if shape.dtype == "f32" else torch.bfloat16


def skewed_router_bias(E: int, gamma: float) -> torch.Tensor:
    """Router logit offsets for the skewed-load workload.

    +2.0 on expert 0 plus Zipf(s=1.1)-shaped log-prior offsets -1.1*ln(e+1),
    both scaled by one constant gamma (the workload names the +2.0 and the
    Zipf exponent but, unscaled, sends every token to expert 0).
    """
    e = torch.arange(E, dtype=torch.float64)
    b = -1.1 * torch.log(e + 1.0)
    b[0] += 2.0
    return (gamma * b).to(torch.float32)


def _normal_(t: torch.Tensor, std: float, gen: torch.Generator) -> None:
    flat = t.view(-1)
    for s in range(0, flat.numel(), _CHUNK_ELEMS):
        part = flat[s:s + _CHUNK_ELEMS]
        tmp = torch.empty(part.shape, dtype=torch.float32, device=t.device)
        tmp.normal_(0.0, std, generator=gen)
        part.copy_(tmp)


def _trunc_normal_(t: torch.Tensor, std: float, gen: torch.Generator) -> None:
    flat = t.view(-1)
    for s in range(0, flat.numel(), _CHUNK_ELEMS):
        part = flat[s:s + _CHUNK_ELEMS]
        tmp = torch.empty(part.shape, dtype=torch.float32, device=t.device)
        torch.nn.init.trunc_normal_(tmp, 0.0, std, -2.0 * std, 2.0 * std, generator=gen)
        part.copy_(tmp)


def make_inputs(shape: LayerShape, seed: int, device="cpu", *, with_experts: bool = True,
                expert_bias_std: float = 0.0, router_bias_std: float = 0.0,
                tie_pairs: int = 0) -> dict:
    """Draw x, router and expert parameters for `shape`.

    Returns a dict of torch tensors on `device`:
      x  [G*T, d]      activations (fp32 or bf16), x ~ N(0, 1)
      Wr [E, d] fp32   router weights, N(0, 0.1/d) or truncated
      br [E] fp32 or None
      W1 [E, d_ff, d], b1 [E, d_ff], W2 [E, d, d_ff], b2 [E, d]  (act dtype)
    Expert and router biases are zero (None) unless a std is given; tests use
    non-zero ones to exercise the bias path.  tie_pairs > 0 copies router row
    2k into row 2k+1 for k < tie_pairs, forcing exact logit ties.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    dt = act_dtype(shape)
    N, d, F, E = shape.N, shape.d_model, shape.d_ff, shape.E

    x = torch.empty(N, d, dtype=dt, device=device)
    _normal_(x, 1.0, gen)

    Wr = torch.empty(E, d, dtype=torch.float32, device=device)
    r_std = math.sqrt(0.1 / d)
    if shape.router_init == "trunc":
        _trunc_normal_(Wr, r_std, gen)
    else:
        _normal_(Wr, r_std, gen)
    for k in range(tie_pairs):
        if 2 * k + 1 < E:
            Wr[2 * k + 1].copy_(Wr[2 * k])

    br: Optional[torch.Tensor] = None
    if shape.router_bias == "skewed":
        br = skewed_router_bias(E, shape.bias_gamma).to(device)
    if router_bias_std > 0.0:
        extra = torch.empty(E, dtype=torch.float32, device=device)
        _normal_(extra, router_bias_std, gen)
        br = extra if br is None else br + extra

    out = {"x": x, "Wr": Wr, "br": br}
    if with_experts:
        W1 = torch.empty(E, F, d, dtype=dt, device=device)
        _trunc_normal_(W1, math.sqrt(0.1 / d), gen)
        W2 = torch.empty(E, d, F, dtype=dt, device=device)
        _trunc_normal_(W2, math.sqrt(0.1 / F), gen)
        b1 = b2 = None
        if expert_bias_std > 0.0:
            b1 = torch.empty(E, F, dtype=dt, device=device)
            _normal_(b1, expert_bias_std, gen)
            b2 = torch.empty(E, d, dtype=dt, device=device)
            _normal_(b2, expert_bias_std, gen)
        out.update(W1=W1, b1=b1, W2=W2, b2=b2)
    return out


def expert_weights(shape: LayerShape, seed: int, expert: int, device="cpu") -> tuple:
    """W1[e] [d_ff, d] and W2[e] [d, d_ff] of one expert, drawn from a generator of its own
    (seed, expert), with make_inputs' distributions but not its values.  For a host-side
    sample that needs a few experts of a layer too large to draw whole on the host."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed) * 65537 + 1 + int(expert))
    dt = act_dtype(shape)
    W1 = torch.empty(shape.d_ff, shape.d_model, dtype=dt, device=device)
    _trunc_normal_(W1, math.sqrt(0.1 / shape.d_model), gen)
    W2 = torch.empty(shape.d_model, shape.d_ff, dtype=dt, device=device)
    _trunc_normal_(W2, math.sqrt(0.1 / shape.d_ff), gen)
    return W1, W2


def workload(name: str) -> LayerShape:
    return WORKLOADS[name]


def workload_seed(name: str) -> int:
    return WORKLOAD_SEEDS[name]
