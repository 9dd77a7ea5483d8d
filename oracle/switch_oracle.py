"""fp64 CPU oracle of the top-1 Switch MoE layer forward pass.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline (and its --impl reference arm) may import or run this module.  The
CUDA library never imports it, and it imports nothing from the library: the two
share no code.  It is deliberately plain and slow: NumPy in float64, one
library matmul per linear map, and pure-Python loops where the pages define a
step as a sequential count.

Pages cited (title, then the section / equation / table):
  [042]  "042 · Switch Transformer：每个词只选一个专家" (wq-win.github.io)
  [card] "Switch Transformers: Scaling to Trillion Parameter Models with Simple
         and Efficient Sparsity - 中文验证版" (ai-papers.xuzou.cn)
  [moe]  "混合专家" (world.lapla.si/zh/moe)
  [070]  "开源 AI 论文复现实验与代码解读 · 070" on MoE routing load collapse
         (zffjzz.top)

Readings taken where the pages leave a step open:
  * argmax is taken over the logits z (softmax is monotone); ties go to the
    lowest expert index, the NumPy rule [070, 核心思想与公式].
  * capacity C = ceil(c*T/E), with c*T/E snapped to an integer when it is within
    1e-9 of one, so that 1.1*100/10 gives 11 [070, 核心思想与公式; 042, §一].
  * f counts choices BEFORE capacity truncation [070, 核心思想与公式].
  * alpha sits inside the loss: L = alpha*E*sum_i f_i P_i [042, §二]; the
    unweighted E*sum f P is returned too.
  * with several routing groups, each group has its own capacity, slots and
    statistics, and the aux loss is the mean over groups [070, 评测协议].
  * the dispatched buffer packs each expert's kept tokens group by group, in
    sequence order: row = (kept tokens of that expert in earlier groups) + slot.
  * y excludes the residual; a dropped token's expert output is exactly 0
    [042, §一; 070, 核心思想与公式 (the m_t mask)].
  * the router z-loss is reported unweighted, per group over that group's T
    tokens, and its mean over groups, like the balance term [070, 核心思想与公式
    (ST-MoE's z-loss) and 最小实验 (both reported without their weights)].
  * top-2 (route_top2): the two highest scores (ties to the lower index), gates =
    softmax over those two scores [moe, 路由器只开两条线]; capacity ceil(2cT/E),
    twice top-1's [card, 方法适配: top-1 about halves the capacity need]; second
    choices take slots after the expert's kept first choices, in sequence order;
    f counts first choices; a dropped choice's weight is not moved to the other.

Every function here is pinned by tests/test_oracle_pins.py against values the
pages print, closed forms, a dense one-hot einsum formulation [card, 方法适配]
and brute force on tiny inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np


def capacity(capacity_factor: float, T: int, E: int, override: int = 0) -> int:
    """Expert capacity per routing group.

    [042, §一]: C is about (T/E)*c; [070, 核心思想与公式] fixes the rounding
    as C = ceil(c*T/E).  `override` > 0 replaces the rule (used to pin the
    [28,12,12,12] -> [8,8,8,8] truncation example).
    """
    if override > 0:
        return int(override)
    if T <= 0 or E <= 0:
        return 0
    v = float(capacity_factor) * T / E
    r = round(v)
    if abs(v - r) <= 1e-9:
        return int(r)
    return int(math.ceil(v))


def router_logits(x: np.ndarray, Wr: np.ndarray, br: Optional[np.ndarray] = None) -> np.ndarray:
    """z_t = W_r x_t (+ b_r), in float64 from the exact input values.

    [042, §一]: p(x) = softmax(W_r x); [070, 核心思想与公式]: Z = X W with W
    of shape [d, E]; here W_r is stored [E, d], so Z = X W_r^T.  The router
    input is cast up before the product [card, 方法适配 (selective precision)].
    """
    z = np.asarray(x, dtype=np.float64) @ np.asarray(Wr, dtype=np.float64).T
    if br is not None:
        z = z + np.asarray(br, dtype=np.float64)[None, :]
    return z


def softmax(z: np.ndarray) -> np.ndarray:
    """Row softmax of the router logits, computed as exp(z - max z) / sum."""
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def top1(z: np.ndarray) -> np.ndarray:
    """e*(x) = argmax_e, first maximal index on ties [042, §一; 070, 核心思想与公式]."""
    return np.argmax(z, axis=-1).astype(np.int64)


def assign_slots(a: Sequence[int], E: int, C: int):
    """Slot of each token inside its expert, in sequence order, and the capacity mask.

    [070, 官方代码阅读路线]: positions come from a cumulative count along the
    sequence, not from an ordering by probability.  Token t's slot is the number
    of earlier tokens of the same group that chose the same expert; the token is
    kept when slot < C [042, §一 (overflow tokens skip the expert)].

    Returns slot [T], keep [T] (bool), raw [E] (choices before truncation) and
    accepted [E] = min(raw, C).
    """
    counts = [0] * E
    T = len(a)
    slot = np.empty(T, dtype=np.int64)
    for t in range(T):
        e = int(a[t])
        slot[t] = counts[e]
        counts[e] += 1
    raw = np.asarray(counts, dtype=np.int64)
    keep = slot < C
    accepted = np.minimum(raw, C)
    return slot, keep, raw, accepted


def load_balance(a: np.ndarray, p: np.ndarray, E: int, alpha: float):
    """f_i, P_i and the auxiliary loss of one routing group.

    [042, §二]: L_aux = alpha * E * sum_e f_e P_e with f_e = (1/T) sum_x 1[e*(x)=e]
    and P_e = (1/T) sum_x p_e(x).  f uses the hard choices before capacity
    truncation [070, 核心思想与公式].
    Returns f [E], P [E], the unweighted term E*sum f P, and alpha times it.
    """
    T = len(a)
    f = np.bincount(np.asarray(a, dtype=np.int64), minlength=E).astype(np.float64) / T
    P = p.mean(axis=0)
    unweighted = E * float(np.sum(f * P))
    return f, P, unweighted, alpha * unweighted


def z_loss(z: np.ndarray) -> float:
    """Router z-loss of one routing group: L_z = (1/T) sum_t (log sum_i exp z_ti)^2.

    [070, 核心思想与公式]: ST-MoE's router z-loss on the score matrix Z (the logits
    before the softmax); it penalises the log normaliser of each token's scores.
    The log-sum-exp is evaluated as m + log sum_i exp(z_ti - m), m = max_i z_ti,
    which is the same number without overflow.
    """
    if z.shape[0] == 0:
        return 0.0
    m = z.max(axis=-1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=-1))
    return float(np.mean(lse * lse))


@dataclasses.dataclass
class Route:
    C: int
    logits: np.ndarray       # [N, E] float64 (or the substituted logits)
    probs: np.ndarray        # [N, E]
    expert: np.ndarray       # [N] raw choice, also for dropped tokens
    gate: np.ndarray         # [N] p_{t, expert_t}
    slot: np.ndarray         # [N]
    keep: np.ndarray         # [N] bool
    row: np.ndarray          # [N] row in the expert's block of xe, -1 if dropped
    raw: np.ndarray          # [G, E]
    accepted: np.ndarray     # [G, E]
    f: np.ndarray            # [G, E]
    P: np.ndarray            # [G, E]
    balance: np.ndarray      # [G] unweighted E * sum f P
    aux_per_group: np.ndarray  # [G] alpha * balance
    aux_loss: float          # mean over groups
    expert_rows: np.ndarray  # [E] kept tokens per expert, all groups
    z_per_group: np.ndarray = None  # [G] router z-loss of each group (unweighted)
    z_loss: float = 0.0             # mean over groups

    @property
    def overflow(self) -> int:
        return int((~self.keep).sum())


def _choice_scores(z: np.ndarray, choice_logits: Optional[dict], T: int) -> np.ndarray:
    """The scores the choice step ranks: z, with the given groups' rows replaced."""
    if not choice_logits:
        return z
    zc = z.copy()
    for g, zg in choice_logits.items():
        zc[g * T:(g + 1) * T] = np.asarray(zg, dtype=np.float64)
    return zc


def route(x, Wr, br, G: int, T: int, E: int, capacity_factor: float, alpha: float = 1e-2,
          capacity_override: int = 0, choice_logits: Optional[dict] = None) -> Route:
    """Router, top-1 choice, slots, capacity mask and load statistics per group.

    Steps in the order of the pipeline in [042, §三]: router probabilities in
    float (here float64), one expert per token, load statistics and aux loss,
    then capacity truncation.

    `choice_logits` maps a group index to a [T, E] array of logits from which
    that group's expert choices are taken instead of from the float64 logits.
    Only the choice step reads it: it decides which expert each token goes to,
    hence slots, capacity mask and the counts f, while the probabilities, the
    gate values p_{t, e*} of the chosen experts, P and the z-loss stay float64.
    It is used where another implementation's float32 logits of a token sit
    within 1e-6 of a tie, so that rounding, not the method, picked between the
    two experts ([070, 核心思想与公式]: the tie rule decides the choice only).
    """
    x = np.asarray(x)
    N = G * T
    assert x.shape[0] == N
    C = capacity(capacity_factor, T, E, capacity_override)
    z = router_logits(x, Wr, br)
    zc = _choice_scores(z, choice_logits, T)
    p = softmax(z) if N > 0 else np.zeros((0, E))
    a = top1(zc) if N > 0 else np.zeros(0, dtype=np.int64)
    gate = p[np.arange(N), a] if N > 0 else np.zeros(0)

    slot = np.empty(N, dtype=np.int64)
    keep = np.empty(N, dtype=bool)
    raw = np.zeros((G, E), dtype=np.int64)
    accepted = np.zeros((G, E), dtype=np.int64)
    f = np.zeros((G, E))
    P = np.zeros((G, E))
    balance = np.zeros(G)
    aux = np.zeros(G)
    zg = np.zeros(G)
    for g in range(G):
        sl = slice(g * T, (g + 1) * T)
        slot[sl], keep[sl], raw[g], accepted[g] = assign_slots(a[sl], E, C)
        if T > 0:
            f[g], P[g], balance[g], aux[g] = load_balance(a[sl], p[sl], E, alpha)
            zg[g] = z_loss(z[sl])

    # Row of each kept token in its expert's block: kept tokens of the same
    # expert in earlier groups come first, then this group's slot.
    row = np.full(N, -1, dtype=np.int64)
    before = np.zeros(E, dtype=np.int64)
    for g in range(G):
        for t in range(g * T, (g + 1) * T):
            if keep[t]:
                row[t] = before[a[t]] + slot[t]
        before += accepted[g]
    return Route(C=C, logits=z, probs=p, expert=a, gate=gate, slot=slot, keep=keep, row=row,
                 raw=raw, accepted=accepted, f=f, P=P, balance=balance, aux_per_group=aux,
                 aux_loss=float(aux.mean()) if G > 0 else 0.0, expert_rows=accepted.sum(axis=0),
                 z_per_group=zg, z_loss=float(zg.mean()) if G > 0 else 0.0)


def dispatch(x, r: Route, E: int, G: int) -> np.ndarray:
    """Gather kept tokens into the per-expert buffer xe [E, G*C, d] (float64).

    [042, §三] builds dispatch tensors after capacity truncation; [card,
    方法适配] writes the dispatch as a one-hot tensor over (tokens, experts,
    capacity), so unused slots hold zeros.  Here each expert's block holds its
    kept tokens group by group in sequence order (see module header).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[1]
    xe = np.zeros((E, G * r.C, d))
    for t in range(x.shape[0]):
        if r.keep[t]:
            xe[r.expert[t], r.row[t]] = x[t]
    return xe


def expert_ffn(xrows, W1, b1, W2, b2) -> np.ndarray:
    """One expert's FFN on rows: ReLU(x W1^T + b1) W2^T + b2, float64.

    [moe, 专家里面是什么]: an expert is an ordinary feed-forward block, d ->
    d_ff with negatives set to 0, then back to d; its parameter count
    (48*32+32+32*48+48 = 3,152) shows both layers carry a bias.
    W1 is stored [d_ff, d] and W2 [d, d_ff].
    """
    xr = np.asarray(xrows, dtype=np.float64)
    h = xr @ np.asarray(W1, dtype=np.float64).T
    if b1 is not None:
        h = h + np.asarray(b1, dtype=np.float64)[None, :]
    h = np.maximum(h, 0.0)
    o = h @ np.asarray(W2, dtype=np.float64).T
    if b2 is not None:
        o = o + np.asarray(b2, dtype=np.float64)[None, :]
    return o


def expert_outputs(x, r: Route, W1, b1, W2, b2, tokens: Optional[Sequence[int]] = None) -> dict:
    """Ungated expert output o_t = f_{e*(t)}(x_t) for kept tokens (or the given subset)."""
    x = np.asarray(x)
    idx = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    idx = idx[r.keep[idx]]
    out = {}
    for e in np.unique(r.expert[idx]):
        sel = idx[r.expert[idx] == e]
        o = expert_ffn(x[sel], W1[e], None if b1 is None else b1[e],
                       W2[e], None if b2 is None else b2[e])
        for i, t in enumerate(sel):
            out[int(t)] = o[i]
    return out


def combine(r: Route, outputs: dict, tokens: Sequence[int], d: int) -> np.ndarray:
    """y_t = p_{e*}(x_t) * f_{e*}(x_t) for kept tokens, 0 for dropped ones.

    [042, §一]: y = p_{e*(x)}(x) f_{e*(x)}(x); the selected gate multiplies the
    expert output un-renormalised ([042], section 只执行一个专家时检查路由是否被错误归一化:
    a gate of 0.7 stays 0.7).  Dropped tokens get zero expert output and carry
    on through the residual, which is outside y [042, §一].
    """
    y = np.zeros((len(tokens), d))
    for i, t in enumerate(tokens):
        if r.keep[t]:
            y[i] = r.gate[t] * outputs[int(t)]
    return y


def forward(x, Wr, br, W1, b1, W2, b2, G: int, T: int, E: int, capacity_factor: float,
            alpha: float = 1e-2, capacity_override: int = 0,
            tokens: Optional[Sequence[int]] = None, choice_logits: Optional[dict] = None):
    """The whole layer: route, then expert FFN and combine on `tokens` (default: all).

    Returns (route, y[tokens], ungated expert outputs by token).
    """
    r = route(x, Wr, br, G, T, E, capacity_factor, alpha, capacity_override, choice_logits)
    N = G * T
    toks = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)
    outs = expert_outputs(x, r, W1, b1, W2, b2, toks)
    y = combine(r, outs, toks, np.asarray(x).shape[1])
    return r, y, outs


def ties_within(z: np.ndarray, eps: float) -> np.ndarray:
    """Per token: True when the two largest logits differ by at most eps."""
    if z.shape[1] < 2:
        return np.zeros(z.shape[0], dtype=bool)
    top2 = np.partition(z, -2, axis=1)[:, -2:]
    return (top2[:, 1] - top2[:, 0]) <= eps


def groups_with_near_ties(z_list: List[np.ndarray], G: int, T: int, eps: float = 1e-6) -> List[int]:
    """Groups in which any token's top-two logits (in any of the given logit
    arrays) lie within eps; such groups are routed from the GPU's own logits."""
    out = []
    for g in range(G):
        sl = slice(g * T, (g + 1) * T)
        if any(ties_within(np.asarray(z, dtype=np.float64)[sl], eps).any() for z in z_list):
            out.append(g)
    return out


# ----------------------------------------------------------------------------- top-2 variant

@dataclasses.dataclass
class Route2:
    C: int
    logits: np.ndarray      # [N, E]
    probs: np.ndarray       # [N, E] full softmax (for P)
    expert: np.ndarray      # [N] first choice
    expert2: np.ndarray     # [N] second choice
    gate: np.ndarray        # [N] weight of the first choice (softmax over the two scores)
    gate2: np.ndarray       # [N] weight of the second choice; gate + gate2 = 1
    slot: np.ndarray        # [N]
    slot2: np.ndarray       # [N] counted after the expert's kept first choices
    keep: np.ndarray        # [N] bool
    keep2: np.ndarray       # [N] bool
    row: np.ndarray         # [N] row in the expert block, -1 if dropped
    row2: np.ndarray        # [N]
    raw: np.ndarray         # [G, E] first choices
    raw2: np.ndarray        # [G, E] second choices
    accepted: np.ndarray    # [G, E] kept first choices
    accepted2: np.ndarray   # [G, E] kept second choices
    f: np.ndarray           # [G, E] first-choice fractions
    P: np.ndarray           # [G, E]
    balance: np.ndarray     # [G]
    aux_per_group: np.ndarray
    aux_loss: float
    z_per_group: np.ndarray
    z_loss: float
    expert_rows: np.ndarray  # [E] kept first + second choices, all groups


def top2(z: np.ndarray):
    """First and second choice: the highest score, then the highest of the others; ties go
    to the lower expert index [moe, 路由器只开两条线 (keep the k highest scores)]."""
    a1 = np.argmax(z, axis=-1).astype(np.int64)
    zz = z.copy()
    zz[np.arange(z.shape[0]), a1] = -np.inf
    a2 = np.argmax(zz, axis=-1).astype(np.int64)
    return a1, a2


def route_top2(x, Wr, br, G: int, T: int, E: int, capacity_factor: float, alpha: float = 1e-2,
               capacity_override: int = 0, choice_logits: Optional[dict] = None) -> Route2:
    """Top-2 routing per group: choices, gates, slots, capacity mask and statistics.

    Gates: softmax over the two kept scores, so they add to 1 [moe, 路由器只开两条线].
    Capacity: ceil(2 c T / E), twice the top-1 capacity [card, 方法适配].  Slots: the
    first choices of the group in sequence order, then its second choices in sequence
    order, each expert's second choices numbered after its kept first choices.
    `choice_logits` (as in `route`) decides the two choices of the given groups; the
    gates are then the softmax over the two chosen experts' float64 scores.
    """
    assert E >= 2
    x = np.asarray(x)
    N = G * T
    C = capacity(2.0 * capacity_factor, T, E, capacity_override)
    z = router_logits(x, Wr, br)
    zc = _choice_scores(z, choice_logits, T)
    p = softmax(z) if N > 0 else np.zeros((0, E))
    a1, a2 = top2(zc) if N > 0 else (np.zeros(0, np.int64), np.zeros(0, np.int64))
    z1 = z[np.arange(N), a1] if N > 0 else np.zeros(0)
    z2 = z[np.arange(N), a2] if N > 0 else np.zeros(0)
    gate = 1.0 / (1.0 + np.exp(z2 - z1))       # exp(z1) / (exp(z1) + exp(z2))
    gate2 = 1.0 / (1.0 + np.exp(z1 - z2))

    slot = np.empty(N, dtype=np.int64)
    slot2 = np.empty(N, dtype=np.int64)
    keep = np.empty(N, dtype=bool)
    keep2 = np.empty(N, dtype=bool)
    raw = np.zeros((G, E), dtype=np.int64)
    raw2 = np.zeros((G, E), dtype=np.int64)
    accepted = np.zeros((G, E), dtype=np.int64)
    accepted2 = np.zeros((G, E), dtype=np.int64)
    f = np.zeros((G, E))
    P = np.zeros((G, E))
    balance = np.zeros(G)
    aux = np.zeros(G)
    zg = np.zeros(G)
    for g in range(G):
        sl = slice(g * T, (g + 1) * T)
        slot[sl], keep[sl], raw[g], accepted[g] = assign_slots(a1[sl], E, C)
        # second choices: numbered per expert in sequence order, after the kept first choices
        s2, _, raw2[g], _ = assign_slots(a2[sl], E, C)
        slot2[sl] = s2 + accepted[g][a2[sl]]
        keep2[sl] = slot2[sl] < C
        accepted2[g] = np.minimum(raw2[g], np.maximum(C - accepted[g], 0))
        if T > 0:
            f[g], P[g], balance[g], aux[g] = load_balance(a1[sl], p[sl], E, alpha)
            zg[g] = z_loss(z[sl])

    row = np.full(N, -1, dtype=np.int64)
    row2 = np.full(N, -1, dtype=np.int64)
    before = np.zeros(E, dtype=np.int64)
    for g in range(G):
        for t in range(g * T, (g + 1) * T):
            if keep[t]:
                row[t] = before[a1[t]] + slot[t]
            if keep2[t]:
                row2[t] = before[a2[t]] + slot2[t]
        before += accepted[g] + accepted2[g]
    return Route2(C=C, logits=z, probs=p, expert=a1, expert2=a2, gate=gate, gate2=gate2, slot=slot, slot2=slot2,
                  keep=keep, keep2=keep2, row=row, row2=row2, raw=raw, raw2=raw2, accepted=accepted,
                  accepted2=accepted2, f=f, P=P, balance=balance, aux_per_group=aux,
                  aux_loss=float(aux.mean()) if G > 0 else 0.0, z_per_group=zg,
                  z_loss=float(zg.mean()) if G > 0 else 0.0,
                  expert_rows=(accepted + accepted2).sum(axis=0))


def combine_top2(r: Route2, outputs: dict, tokens: Sequence[int], d: int) -> np.ndarray:
    """y_t = sum over the token's kept choices of gate_k * FFN_{e_k}(x_t)
    [moe, 路由器只开两条线: the two results are added with their weights]; 0 when both
    choices are dropped.  `outputs` maps (token, expert) to that expert's output row."""
    y = np.zeros((len(tokens), d))
    for i, t in enumerate(tokens):
        if r.keep[t]:
            y[i] += r.gate[t] * outputs[(t, int(r.expert[t]))]
        if r.keep2[t]:
            y[i] += r.gate2[t] * outputs[(t, int(r.expert2[t]))]
    return y


def forward_top2(x, Wr, br, W1, b1, W2, b2, G: int, T: int, E: int, capacity_factor: float,
                 tokens: Optional[Sequence[int]] = None, alpha: float = 1e-2, capacity_override: int = 0):
    """The top-2 layer on `tokens` (all when None): returns (y rows, Route2)."""
    r = route_top2(x, Wr, br, G, T, E, capacity_factor, alpha, capacity_override)
    tokens = list(range(G * T)) if tokens is None else list(tokens)
    return combine_top2(r, expert_outputs_top2(x, r, W1, b1, W2, b2, tokens), tokens, np.asarray(x).shape[1]), r


def expert_outputs_top2(x, r: Route2, W1, b1, W2, b2, tokens: Optional[Sequence[int]] = None) -> dict:
    """Ungated outputs FFN_e(x_t) for every kept (token, choice): {(t, e): row}."""
    x = np.asarray(x)
    idx = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = {}
    for ex, kp in ((r.expert, r.keep), (r.expert2, r.keep2)):
        sel_all = idx[kp[idx]]
        for e in np.unique(ex[sel_all]):
            sel = sel_all[ex[sel_all] == e]
            o = expert_ffn(x[sel], W1[e], None if b1 is None else b1[e], W2[e], None if b2 is None else b2[e])
            for i, t in enumerate(sel):
                out[(int(t), int(e))] = o[i]
    return out


# ----------------------------------------------------------------------------- expert parallelism

def ep_forward(x_ranks, Wr, br, W1, b1, W2, b2, G: int, T: int, E: int, capacity_factor: float, world: int,
               alpha: float = 1e-2, capacity_override: int = 0):
    """The top-1 layer with its experts sharded over `world` ranks, step by step.

    [card, 方法适配]: the input is laid out per core, every core routes its own tokens, an
    all-to-all sends each token to the core holding its expert, the experts run there, and a
    second all-to-all returns the outputs for the combine.  Reading: rank r holds the experts
    floor(rE/world) .. floor((r+1)E/world) - 1 and routes its own G groups of T tokens
    (x_ranks[r] is [G*T, d]); what travels is each rank's per-expert block of the dispatched
    buffer with its valid row count.  Written with explicit per-rank send and receive lists
    (no communication library).  Returns (routes per rank, y per rank).
    """
    begin = [(r * E) // world for r in range(world + 1)]
    routes, xe = [], []
    for r in range(world):
        rt = route(x_ranks[r], Wr, br, G, T, E, capacity_factor, alpha, capacity_override)
        routes.append(rt)
        xe.append(dispatch(x_ranks[r], rt, E, G))  # [E, G*C, d]
    # first all-to-all: owner o receives from every source s the blocks of its experts
    recv = [[xe[s][begin[o]:begin[o + 1]] for s in range(world)] for o in range(world)]
    rows = [[routes[s].expert_rows[begin[o]:begin[o + 1]] for s in range(world)] for o in range(world)]
    # each owner runs its experts on the rows received from all sources
    out = [[np.zeros_like(recv[o][s]) for s in range(world)] for o in range(world)]
    for o in range(world):
        for j, e in enumerate(range(begin[o], begin[o + 1])):
            parts = [recv[o][s][j, :int(rows[o][s][j])] for s in range(world)]
            stacked = np.concatenate(parts, axis=0)
            if stacked.shape[0] == 0:
                continue
            ye = expert_ffn(stacked, W1[e], None if b1 is None else b1[e], W2[e], None if b2 is None else b2[e])
            at = 0
            for s in range(world):
                n = int(rows[o][s][j])
                out[o][s][j, :n] = ye[at:at + n]
                at += n
    # second all-to-all: source s gets back the output blocks of every owner, in expert order
    ye_back = [np.concatenate([out[o][s] for o in range(world)], axis=0) for s in range(world)]
    ys = []
    for s in range(world):
        rt = routes[s]
        y = np.zeros((G * T, np.asarray(x_ranks[s]).shape[1]))
        for t in range(G * T):
            if rt.keep[t]:
                y[t] = rt.gate[t] * ye_back[s][rt.expert[t], rt.row[t]]
        ys.append(y)
    return routes, ys


# ----------------------------------------------------------------------------- backward (top-1)

def backward(x, Wr, br, W1, b1, W2, b2, G: int, T: int, E: int, capacity_factor: float, dy,
             w_aux: float = 0.0, w_z: float = 0.0, alpha: float = 1e-2, capacity_override: int = 0,
             residual: bool = False, choice_logits: Optional[dict] = None) -> dict:
    """Gradients of L = sum(dy * y) + w_aux * aux_loss + w_z * z_loss for the top-1 layer.

    The choice, the slots and the capacity mask are held fixed (they are piecewise
    constant): the router gets its gradient through the selected expert's probability g_t =
    p_{t,e*} [card, 方法适配: the gate probability keeps the router differentiable] and
    through P in the aux loss, not through the hard counts f [070, 核心思想与公式]; the
    z-loss adds d(lse_t^2)/dz = 2 lse_t p_t [070, 核心思想与公式].  With several groups the
    aux and z losses are means over groups.  Returns float64 arrays: dx [N, d], dWr [E, d],
    dbr [E], dW1 [E, F, d], db1 [E, F], dW2 [E, d, F], db2 [E, d].
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    N, d = x.shape
    F = W1.shape[1]
    r = route(x, Wr, br, G, T, E, capacity_factor, alpha, capacity_override, choice_logits)
    p = r.probs
    dx = dy.copy() if residual else np.zeros_like(x)
    dW1 = np.zeros_like(W1)
    dW2 = np.zeros_like(W2)
    db1 = np.zeros((E, F))
    db2 = np.zeros((E, d))
    dg = np.zeros(N)
    # experts: y_t = g_t * (ReLU(x_t W1^T + b1) W2^T + b2) for kept tokens
    for e in range(E):
        ts = np.flatnonzero(r.keep & (r.expert == e))
        if ts.size == 0:
            continue
        xe = x[ts]
        hpre = xe @ W1[e].T + (0.0 if b1 is None else np.asarray(b1, np.float64)[e])
        h = np.maximum(hpre, 0.0)
        o = h @ W2[e].T + (0.0 if b2 is None else np.asarray(b2, np.float64)[e])
        dg[ts] = np.sum(dy[ts] * o, axis=1)
        do = r.gate[ts, None] * dy[ts]                 # dL/d(expert output)
        dW2[e] = do.T @ h
        db2[e] = do.sum(axis=0)
        dh = (do @ W2[e]) * (hpre > 0)
        dW1[e] = dh.T @ xe
        db1[e] = dh.sum(axis=0)
        dx[ts] += dh @ W1[e]
    # router: dL/dp, then the softmax Jacobian, plus the z-loss term on the logits
    dp = np.zeros_like(p)
    dp[np.arange(N), r.expert] = dg
    dz = np.zeros_like(p)
    for g in range(G):
        sl = slice(g * T, (g + 1) * T)
        if T == 0:
            continue
        dp[sl] += (w_aux * alpha * E / (G * T)) * r.f[g][None, :]
        ps = p[sl]
        dz[sl] = ps * (dp[sl] - np.sum(ps * dp[sl], axis=1, keepdims=True))
        zg = r.logits[sl]
        m = zg.max(axis=1, keepdims=True)
        lse = m + np.log(np.exp(zg - m).sum(axis=1, keepdims=True))
        dz[sl] += (w_z * 2.0 / (G * T)) * lse * ps
    dWr = dz.T @ x
    dbr = dz.sum(axis=0)
    dx += dz @ Wr
    return dict(dx=dx, dWr=dWr, dbr=dbr, dW1=dW1, db1=db1, dW2=dW2, db2=db2, route=r)
