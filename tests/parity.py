"""Helpers that run the CUDA layer through the C ABI and compare it with the fp64 oracle.

Comparison rules:
  * expert, slot, keep, row, raw/accepted counts, expert rows: bit-exact;
  * gate, probabilities, P, balance, aux loss and router z-loss: |a - b| <= 1e-5 * |b|;
  * dispatched rows: bit-exact copies of x; rows past an expert's count are zero;
  * y: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| elementwise, plus per kept token
    ||y_t - y_ref,t|| <= 1e-2 ||y_ref,t|| (the elementwise bound alone would pass an
    all-zero output at these init scales), and y_t == 0 exactly for dropped tokens;
  * ungated expert output rows: ||ye_row - o_ref|| <= 1e-2 ||o_ref||.
  * router logits (when written): |z - z_ref| <= 1e-5 on every logit, compared with the
    float64 oracle before anything else.
Near ties: where any token's top-two float32 logits (GPU) or float64 logits
(oracle) lie within 1e-6, the choices of that token's whole group are taken by
the oracle from the GPU's own float32 logits (the oracle's dispatch stage: one
flipped choice shifts every later slot of that expert in the group).  Only the
choices move: probabilities, gates, P, balance, aux and z-loss are still the
float64 oracle's values for every token.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import switch_oracle as so

REL_FLOAT = 1e-5
Y_ATOL, Y_RTOL = 1e-2, 1e-2
ROW_REL_L2 = 1e-2
TIE_EPS = 1e-6
LOGIT_ABS = 1e-5


def to_np(t):
    return None if t is None else t.detach().float().cpu().numpy().astype(np.float64) if t.is_floating_point() \
        else t.detach().cpu().numpy()


def make_layer(shape, **kw):
    from sparse_mixture_experts_slots_b300 import SwitchMoE
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    return SwitchMoE(shape.G, shape.T, shape.d_model, shape.d_ff, shape.E, shape.capacity_factor, dtype=dt,
                     capacity_override=shape.capacity_override, **kw)


def oracle_route(inp, shape, gpu_logits: np.ndarray | None = None):
    """Oracle routing; in groups with near ties the GPU's logits decide the choices.

    Returns (route, substituted group indices)."""
    x = to_np(inp["x"])
    Wr = to_np(inp["Wr"])
    br = to_np(inp["br"]) if inp["br"] is not None else None
    r = so.route(x, Wr, br, shape.G, shape.T, shape.E, shape.capacity_factor,
                 capacity_override=shape.capacity_override)
    subst = []
    if gpu_logits is not None and shape.N > 0:
        subst = so.groups_with_near_ties([gpu_logits, r.logits], shape.G, shape.T, TIE_EPS)
        if subst:
            over = {g: gpu_logits[g * shape.T:(g + 1) * shape.T] for g in subst}
            r = so.route(x, Wr, br, shape.G, shape.T, shape.E, shape.capacity_factor,
                         capacity_override=shape.capacity_override, choice_logits=over)
    return r, subst


def near_tie_tokens(gpu_logits: np.ndarray, ref_logits: np.ndarray) -> int:
    """Tokens whose top-two logits (GPU float32 or oracle float64) lie within TIE_EPS."""
    return int((so.ties_within(gpu_logits, TIE_EPS) | so.ties_within(ref_logits, TIE_EPS)).sum())


def check_logits(gpu_logits: np.ndarray, ref: so.Route, what: str = "logits"):
    """Every float32 logit within LOGIT_ABS of the float64 oracle's (never substituted)."""
    err = np.abs(np.asarray(gpu_logits, dtype=np.float64) - ref.logits)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= LOGIT_ABS, f"{what}: max |z - z_ref| = {worst:.3e} > {LOGIT_ABS}"
    return worst


def rel_close(a, b, rel=REL_FLOAT, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    bad = np.abs(a - b) > rel * np.abs(b)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} beyond rel {rel}; worst "
                           f"{np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-300)):.3e}")


def compare_route(g, ref: so.Route, shape):
    N, G, E = shape.N, shape.G, shape.E
    assert np.array_equal(to_np(g.expert).astype(np.int64), ref.expert), "expert"
    assert np.array_equal(to_np(g.slot).astype(np.int64), ref.slot), "slot"
    assert np.array_equal(to_np(g.keep).astype(bool), ref.keep), "keep"
    assert np.array_equal(to_np(g.row).astype(np.int64), ref.row), "row"
    assert np.array_equal(to_np(g.raw_count).reshape(G, E).astype(np.int64), ref.raw), "raw counts"
    assert np.array_equal(to_np(g.accepted_count).reshape(G, E).astype(np.int64), ref.accepted), "accepted"
    assert np.array_equal(to_np(g.expert_rows).astype(np.int64), ref.expert_rows), "expert rows"
    if N > 0:
        rel_close(to_np(g.gate), ref.gate, what="gate")
        rel_close(to_np(g.P).reshape(G, E), ref.P, what="P")
        rel_close(to_np(g.balance), ref.balance, what="balance")
        rel_close(to_np(g.aux_loss_per_group), ref.aux_per_group, what="aux per group")
        rel_close(to_np(g.aux_loss)[0], ref.aux_loss, what="aux loss")
        if g.z_loss is not None:
            rel_close(to_np(g.z_loss_per_group), ref.z_per_group, what="z-loss per group")
            rel_close(to_np(g.z_loss)[0], ref.z_loss, what="z-loss")
        if g.probs is not None:
            rel_close(to_np(g.probs), ref.probs, what="probs")
    else:
        assert (to_np(g.P) == 0).all() and (to_np(g.aux_loss) == 0).all()
        if g.z_loss is not None:
            assert (to_np(g.z_loss) == 0).all()


def check_dispatch(xe: torch.Tensor, x: torch.Tensor, ref: so.Route):
    """Kept rows are bit-exact copies of x; rows past each expert's count are zero."""
    kept = np.flatnonzero(ref.keep)
    if kept.size:
        e = torch.as_tensor(ref.expert[kept], device=xe.device)
        r = torch.as_tensor(ref.row[kept], device=xe.device)
        t = torch.as_tensor(kept, device=xe.device)
        assert torch.equal(xe[e, r], x[t]), "dispatched rows differ from x"
    rows = torch.as_tensor(ref.expert_rows, device=xe.device)
    idx = torch.arange(xe.shape[1], device=xe.device)[None, :]
    empty = idx >= rows[:, None]
    assert (xe[empty] == 0).all(), "rows past the expert count are not zero"


def sample_tokens(ref: so.Route, n: int, seed: int = 0) -> np.ndarray:
    N = ref.keep.size
    if N <= n:
        return np.arange(N)
    rng = np.random.default_rng(seed)
    kept = np.flatnonzero(ref.keep)
    dropped = np.flatnonzero(~ref.keep)
    pick = list(rng.choice(kept, size=min(len(kept), n - min(len(dropped), n // 8)), replace=False))
    if len(dropped):
        pick += list(rng.choice(dropped, size=min(len(dropped), n // 8), replace=False))
    return np.sort(np.array(pick, dtype=np.int64))


def structured_tokens(ref: so.Route, chunk: int = 256, max_experts: int | None = None, seed: int = 0) -> np.ndarray:
    """Tokens at the edges of each expert block: the rows the FFN's tiling treats apart.

    Per expert (all of them, or `max_experts` of them: a random draw plus the fullest and the
    emptiest non-empty expert), the tokens dispatched to its first and last kept row and to
    the rows on both sides of every `chunk`-row boundary of its block."""
    kept = np.flatnonzero(ref.keep)
    E = ref.expert_rows.size
    experts = np.flatnonzero(ref.expert_rows > 0)
    if max_experts is not None and experts.size > max_experts:
        rng = np.random.default_rng(seed)
        fullest = experts[np.argmax(ref.expert_rows[experts])]
        emptiest = experts[np.argmin(ref.expert_rows[experts])]
        experts = np.unique(np.concatenate([rng.choice(experts, size=max_experts - 2, replace=False),
                                            [fullest, emptiest]]))
    tok_of = {}
    for t in kept:
        e = int(ref.expert[t])
        tok_of.setdefault(e, {})[int(ref.row[t])] = int(t)
    pick = []
    for e in experts:
        n = int(ref.expert_rows[e])
        rows = {0, n - 1}
        for c in range(chunk, n, chunk):
            rows.update((c - 1, c))
        pick += [tok_of[int(e)][r] for r in rows if r in tok_of.get(int(e), {})]
    assert E == 0 or experts.size == 0 or pick, "no kept token found at an expert block edge"
    return np.unique(np.asarray(pick, dtype=np.int64))


def oracle_outputs(inp, ref: so.Route, tokens: np.ndarray) -> dict:
    """Ungated fp64 expert outputs for the kept tokens among `tokens` (weights copied per expert)."""
    x = inp["x"]
    out = {}
    sel = tokens[ref.keep[tokens]]
    for e in np.unique(ref.expert[sel]):
        ts = sel[ref.expert[sel] == e]
        W1 = to_np(inp["W1"][int(e)])
        W2 = to_np(inp["W2"][int(e)])
        b1 = to_np(inp["b1"][int(e)]) if inp["b1"] is not None else None
        b2 = to_np(inp["b2"][int(e)]) if inp["b2"] is not None else None
        o = so.expert_ffn(to_np(x[torch.as_tensor(ts, device=x.device)]), W1, b1, W2, b2)
        for i, t in enumerate(ts):
            out[int(t)] = o[i]
    return out


def check_expert_rows(ye: torch.Tensor, ref: so.Route, outs: dict):
    for t, o in outs.items():
        got = ye[int(ref.expert[t]), int(ref.row[t])].float().cpu().numpy().astype(np.float64)
        err = np.linalg.norm(got - o)
        assert err <= ROW_REL_L2 * np.linalg.norm(o) + 1e-30, f"ye row of token {t}: rel L2 {err / np.linalg.norm(o):.3e}"


def check_y(y: torch.Tensor, ref: so.Route, outs: dict, tokens: np.ndarray, resid: torch.Tensor | None = None):
    yt = to_np(y[torch.as_tensor(tokens, device=y.device)])
    if resid is not None:
        base = to_np(resid[torch.as_tensor(tokens, device=y.device)])
    for i, t in enumerate(tokens):
        yref = ref.gate[t] * outs[int(t)] if ref.keep[t] else np.zeros(yt.shape[1])
        if resid is not None:
            yref = yref + base[i]
        got = yt[i]
        if not ref.keep[t] and resid is None:
            assert (got == 0).all(), f"dropped token {t} has non-zero expert output"
            continue
        bad = np.abs(got - yref) > Y_ATOL + Y_RTOL * np.abs(yref)
        assert not bad.any(), f"token {t}: y outside |y-y_ref| <= 1e-2 + 1e-2|y_ref|"
        if ref.keep[t] and resid is None:  # with a residual the bf16 rounding of x + y dominates
            dref = ref.gate[t] * outs[int(t)]
            err = np.linalg.norm(got - dref)
            assert err <= ROW_REL_L2 * np.linalg.norm(dref) + 1e-30, \
                f"token {t}: y rel L2 {err / np.linalg.norm(dref):.3e}"


# ----------------------------------------------------------------------------- top-2 routing

def top3_near_ties(z: np.ndarray, eps: float) -> np.ndarray:
    """Tokens whose first/second or second/third highest logits lie within eps: rounding
    can swap the two choices' order or change the second choice there."""
    s = -np.sort(-z, axis=1)
    gap = s[:, 0] - s[:, 1]
    if z.shape[1] >= 3:
        gap = np.minimum(gap, s[:, 1] - s[:, 2])
    return gap < eps


def oracle_route_top2(inp, shape, gpu_logits: np.ndarray):
    """Oracle top-2 routing; in groups with a near tie among a token's top three logits (GPU
    or oracle) the GPU's own float32 logits decide the two choices."""
    x = to_np(inp["x"])
    Wr = to_np(inp["Wr"])
    br = to_np(inp["br"]) if inp["br"] is not None else None
    r = so.route_top2(x, Wr, br, shape.G, shape.T, shape.E, shape.capacity_factor,
                      capacity_override=shape.capacity_override)
    subst = []
    if shape.N > 0:
        near = top3_near_ties(gpu_logits, TIE_EPS) | top3_near_ties(r.logits, TIE_EPS)
        subst = sorted({int(t) // shape.T for t in np.flatnonzero(near)})
        if subst:
            over = {g: gpu_logits[g * shape.T:(g + 1) * shape.T] for g in subst}
            r = so.route_top2(x, Wr, br, shape.G, shape.T, shape.E, shape.capacity_factor,
                              capacity_override=shape.capacity_override, choice_logits=over)
    return r, subst


def compare_route_top2(g, ref: so.Route2, shape):
    G, E = shape.G, shape.E
    for name, want in (("expert", ref.expert), ("expert2", ref.expert2), ("slot", ref.slot), ("slot2", ref.slot2),
                       ("row", ref.row), ("row2", ref.row2)):
        assert np.array_equal(to_np(getattr(g, name)).astype(np.int64), want), name
    assert np.array_equal(to_np(g.keep).astype(bool), ref.keep), "keep"
    assert np.array_equal(to_np(g.keep2).astype(bool), ref.keep2), "keep2"
    for name, want in (("raw_count", ref.raw), ("accepted_count", ref.accepted), ("raw2_count", ref.raw2),
                       ("accepted2_count", ref.accepted2)):
        assert np.array_equal(to_np(getattr(g, name)).reshape(G, E).astype(np.int64), want), name
    assert np.array_equal(to_np(g.expert_rows).astype(np.int64), ref.expert_rows), "expert rows"
    if shape.N > 0:
        rel_close(to_np(g.gate), ref.gate, what="gate")
        rel_close(to_np(g.gate2), ref.gate2, what="gate2")
        rel_close(to_np(g.P).reshape(G, E), ref.P, what="P")
        rel_close(to_np(g.balance), ref.balance, what="balance")
        rel_close(to_np(g.aux_loss)[0], ref.aux_loss, what="aux loss")
        rel_close(to_np(g.z_loss_per_group), ref.z_per_group, what="z-loss per group")


def check_dispatch_top2(xe: torch.Tensor, x: torch.Tensor, ref: so.Route2):
    for ex, kp, rw in ((ref.expert, ref.keep, ref.row), (ref.expert2, ref.keep2, ref.row2)):
        kept = np.flatnonzero(kp)
        if kept.size:
            e = torch.as_tensor(ex[kept], device=xe.device)
            r = torch.as_tensor(rw[kept], device=xe.device)
            assert torch.equal(xe[e, r], x[torch.as_tensor(kept, device=xe.device)]), "dispatched rows differ from x"
    rows = torch.as_tensor(ref.expert_rows, device=xe.device)
    idx = torch.arange(xe.shape[1], device=xe.device)[None, :]
    assert (xe[idx >= rows[:, None]] == 0).all(), "rows past the expert count are not zero"


def check_y_top2(y: torch.Tensor, ref: so.Route2, inp, tokens: np.ndarray, resid: torch.Tensor | None = None):
    """y against the oracle's weighted pair of fp64 expert outputs (the elementwise bound, and
    a per-token relative L2 bound where some choice was kept and there is no residual)."""
    xs = {k: (to_np(v) if v is not None else None) for k, v in inp.items() if k in ("W1", "b1", "W2", "b2")}
    outs = so.expert_outputs_top2(to_np(inp["x"]), ref, xs["W1"], xs["b1"], xs["W2"], xs["b2"], tokens)
    yref_all = so.combine_top2(ref, outs, tokens, y.shape[1])
    yt = to_np(y[torch.as_tensor(tokens, device=y.device)])
    base = to_np(resid[torch.as_tensor(tokens, device=y.device)]) if resid is not None else None
    for i, t in enumerate(tokens):
        yref = yref_all[i] + (base[i] if base is not None else 0.0)
        got = yt[i]
        any_kept = ref.keep[t] or ref.keep2[t]
        if not any_kept and resid is None:
            assert (got == 0).all(), f"token {t} with both choices dropped has non-zero output"
            continue
        bad = np.abs(got - yref) > Y_ATOL + Y_RTOL * np.abs(yref)
        assert not bad.any(), f"token {t}: y outside |y-y_ref| <= 1e-2 + 1e-2|y_ref|"
        if any_kept and resid is None:
            err = np.linalg.norm(got - yref)
            assert err <= ROW_REL_L2 * np.linalg.norm(yref) + 1e-30, \
                f"token {t}: y rel L2 {err / np.linalg.norm(yref):.3e}"
