"""Pins for the fp64 oracle: values the pages print, closed forms, and brute force.

Every check here is independent of the oracle's own code path: it uses numbers
printed on the pages (tests/golden/*.json, each citing its source), closed forms,
or a second formulation written out in this file (the dense one-hot einsum of
the Mesh-TensorFlow dispatch/combine, a cumulative-sum slot rule, triple loops).
"""
import math

import numpy as np
import pytest

from oracle import switch_oracle as so
from gen import WORKLOADS


# ----------------------------------------------------------------------------- helpers

def logits_from_p0(q):
    """Scalar input whose two-expert logits [x, 0] give p_0 = q (x = logit(q))."""
    return math.log(q / (1.0 - q))


def two_expert_router():
    # d = 1, E = 2: z = [x, 0]  -> p_0 = sigmoid(x)
    return np.array([[1.0], [0.0]])


def cumsum_slots(a, E):
    """Slots as the Mesh-TF code computes them: cumulative sum of the one-hot
    choice mask along the sequence, minus one, read at the chosen expert."""
    a = np.asarray(a)
    mask = np.zeros((len(a), E), dtype=np.int64)
    mask[np.arange(len(a)), a] = 1
    pos = np.cumsum(mask, axis=0) - 1
    return pos[np.arange(len(a)), a]


def dense_einsum_forward(x, Wr, br, W1, b1, W2, b2, G, T, E, C):
    """Brute force: one-hot dispatch tensor D[g,t,e,c], combine = D * p, every
    expert evaluated on every token, y = einsum over (e, c).  Mirrors the
    dispatch/combine tensor formulation on the xuzou.cn Switch Transformers card
    (section 方法适配)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[1]
    z = x @ np.asarray(Wr, np.float64).T + (0 if br is None else np.asarray(br, np.float64))
    zmax = z.max(axis=1, keepdims=True)
    p = np.exp(z - zmax)
    p /= p.sum(axis=1, keepdims=True)
    a = np.array([min(np.flatnonzero(row == row.max())) for row in z])
    D = np.zeros((G, T, E, max(C, 1)))
    for g in range(G):
        pos = cumsum_slots(a[g * T:(g + 1) * T], E)
        for t in range(T):
            if pos[t] < C:
                D[g, t, a[g * T + t], pos[t]] = 1.0
    comb = D * p.reshape(G, T, E)[..., None]
    # all experts on all tokens
    W1d, W2d = np.asarray(W1, np.float64), np.asarray(W2, np.float64)
    h = np.einsum("nd,efd->nef", x, W1d)
    if b1 is not None:
        h = h + np.asarray(b1, np.float64)[None]
    h = np.maximum(h, 0)
    o = np.einsum("nef,edf->ned", h, W2d)
    if b2 is not None:
        o = o + np.asarray(b2, np.float64)[None]
    y = np.einsum("gtec,gted->gtd", comb, o.reshape(G, T, E, d)).reshape(G * T, d)
    xe_groups = np.einsum("gtec,gtd->gecd", D, x.reshape(G, T, d))
    return y, D, xe_groups, a, p


# ----------------------------------------------------------------------------- capacity

def test_capacity_rule_closed_forms():
    # ceil(c*T/E) [070, 核心思想与公式]; 1.1*100/10 is 11.000000000000002 in binary
    assert so.capacity(1.0, 32, 16) == 2
    assert so.capacity(1.0, 8192, 128) == 64
    assert so.capacity(1.25, 4096, 64) == 80
    assert so.capacity(1.25, 32768, 128) == 320
    assert so.capacity(1.0, 65536, 2048) == 32
    assert so.capacity(1.1, 100, 10) == 11
    assert so.capacity(1.0, 10, 3) == 4
    assert so.capacity(0.5, 64, 4) == 8
    assert so.capacity(1.0, 7, 8) == 1
    assert so.capacity(2.0, 0, 4) == 0
    assert so.capacity(1.0, 64, 4, override=8) == 8


def test_workload_capacities():
    want = {"tiny-e16-fp32": 2, "switch-base-e128": 64, "skewed-e64-g8": 80,
            "switch-large-e128": 320, "many-experts-e2048": 32}
    for name, C in want.items():
        s = WORKLOADS[name]
        assert so.capacity(s.capacity_factor, s.T, s.E) == C


# ----------------------------------------------------------------------------- aux loss

def test_aux_worked_example_1_48(golden):
    g = golden("aux_two_experts.json")
    # Realise f=(0.9, 0.1), P=(0.8, 0.2) with tokens: 9 tokens at p0 = 7.8/9, one at 0.2.
    q_hi, q_lo = 7.8 / 9.0, 0.2
    x = np.array([[logits_from_p0(q_hi)]] * 9 + [[logits_from_p0(q_lo)]])
    r = so.route(x, two_expert_router(), None, G=1, T=10, E=2, capacity_factor=10.0, alpha=0.01)
    np.testing.assert_allclose(r.f[0], g["f"], atol=1e-15)
    np.testing.assert_allclose(r.P[0], g["P"], atol=1e-12)
    assert abs(r.balance[0] - g["balance"]) < 1e-12
    assert abs(r.aux_loss - 0.01 * g["balance"]) < 1e-14
    # direct formula on the printed numbers
    f, P = np.array(g["f"]), np.array(g["P"])
    assert abs(g["E"] * np.sum(f * P) - g["balance"]) < 1e-12


def test_aux_perfect_balance_is_one(golden):
    g = golden("aux_two_experts.json")
    E, T = 4, 8
    x = np.zeros((T, E))
    x[np.arange(T), np.arange(T) % E] = 1.0
    Wr = 3.0 * np.eye(E)  # token t strongly prefers expert t % E, symmetric rows
    r = so.route(x, Wr, None, G=1, T=T, E=E, capacity_factor=1.0)
    np.testing.assert_allclose(r.f[0], 0.25)
    np.testing.assert_allclose(r.P[0], 0.25, atol=1e-15)
    assert abs(r.balance[0] - g["balance_perfect"]) < 1e-12


def test_uniform_probabilities_all_pick_expert0(golden):
    g = golden("uniform_probs_overflow.json")
    rng = np.random.default_rng(0)
    T, E = g["T"], g["E"]
    x = rng.standard_normal((T, 5))
    Wr = np.zeros((E, 5))
    r = so.route(x, Wr, None, G=1, T=T, E=E, capacity_factor=g["capacity_factor"])
    np.testing.assert_allclose(r.probs, 0.25)
    assert (r.expert == g["expert_all"]).all()
    np.testing.assert_allclose(r.f[0], g["f"])
    assert abs(r.balance[0] - g["balance"]) < 1e-12
    assert r.C == g["C"]
    assert r.accepted[0].tolist() == g["accepted"]
    assert r.raw[0].tolist() == [T, 0, 0, 0]
    assert r.overflow / T == pytest.approx(g["overflow_fraction"], abs=0)


def test_truncation_to_equal_accepted(golden):
    g = golden("truncation_equal_accepted.json")
    raw = g["raw"]
    E, T = len(raw), sum(raw)
    # interleave the choices so truncation cuts each expert in sequence order
    a = np.concatenate([np.full(n, e) for e, n in enumerate(raw)])
    rng = np.random.default_rng(1)
    a = a[rng.permutation(T)]
    x = np.zeros((T, E))
    x[np.arange(T), a] = 1.0
    Wr = 4.0 * np.eye(E)
    for kw in ({"capacity_override": g["C"], "capacity_factor": 1.0},
               {"capacity_factor": 0.5}):  # ceil(0.5*64/4) = 8 as well
        r = so.route(x, Wr, None, G=1, T=T, E=E, **kw)
        assert r.C == g["C"]
        assert r.raw[0].tolist() == raw
        assert r.accepted[0].tolist() == g["accepted"]
        # f counts the raw choices, not the accepted ones
        np.testing.assert_allclose(r.f[0], np.array(raw) / T)
        # the kept ones are the first C of each expert in sequence order
        for e in range(E):
            idx = np.flatnonzero(a == e)
            assert r.keep[idx[:g["C"]]].all() and not r.keep[idx[g["C"]:]].any()


def test_shift_invariance_plus_100(golden):
    g = golden("shift_invariance.json")
    rng = np.random.default_rng(2)
    T, E, d = 50, 6, 7
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d)) * 0.3
    br = rng.standard_normal(E) * 0.1
    r0 = so.route(x, Wr, br, 1, T, E, 1.0)
    r1 = so.route(x, Wr, br + g["shift"], 1, T, E, 1.0)
    np.testing.assert_allclose(r1.probs, r0.probs, rtol=1e-12, atol=1e-15)
    assert (r1.expert == r0.expert).all()
    assert (r1.slot == r0.slot).all() and (r1.keep == r0.keep).all()
    # and the max-subtracted softmax does not overflow for large logits
    p = so.softmax(np.array([[1000.0, 999.0]]))
    np.testing.assert_allclose(p, [[1 / (1 + math.exp(-1)), 1 / (1 + math.exp(1))]], rtol=1e-14)


def test_softmax_two_experts_is_sigmoid():
    for v in (-3.0, -0.2, 0.0, 0.5, 4.0):
        p = so.softmax(np.array([[v, 0.0]]))
        assert abs(p[0, 0] - 1.0 / (1.0 + math.exp(-v))) < 1e-15
        assert abs(p.sum() - 1.0) < 1e-15


# ----------------------------------------------------------------------------- gate / combine

def test_gate_not_renormalised(golden):
    g = golden("gate_not_renormalised.json")
    q = g["p_selected"]
    x = np.array([[logits_from_p0(q)]])
    W1 = np.array([[[2.0]], [[-1.0]]])   # E=2, d_ff=1, d=1
    W2 = np.array([[[3.0]], [[5.0]]])
    b1 = np.array([[0.5], [0.0]])
    b2 = np.array([[0.25], [0.0]])
    r, y, outs = so.forward(x, two_expert_router(), None, W1, b1, W2, b2, G=1, T=1, E=2,
                            capacity_factor=2.0)
    assert r.expert[0] == 0
    assert abs(r.gate[0] - g["gate"]) < 1e-15
    o = max(0.0, 2.0 * x[0, 0] + 0.5) * 3.0 + 0.25
    assert abs(outs[0][0] - o) < 1e-14
    assert abs(y[0, 0] - g["gate"] * o) < 1e-14
    assert abs(y[0, 0] - o) > 0.1  # a renormalised gate (=1) would give o


def test_local_overflow_with_enough_total_capacity(golden):
    g = golden("local_overflow.json")
    T, E, A = g["T"], g["E"], 3
    a = [A] * g["tokens_to_A"]
    others = [e for e in range(E) if e != A]
    for i in range(T - g["tokens_to_A"]):
        a.append(others[i % len(others)])  # 70 tokens over 9 experts: at most 8 each
    a = np.array(a)[np.random.default_rng(3).permutation(T)]
    x = np.zeros((T, E))
    x[np.arange(T), a] = 1.0
    r = so.route(x, 5.0 * np.eye(E), None, 1, T, E, g["capacity_factor"])
    assert r.C == g["C"] and E * r.C == T
    assert r.accepted[0, A] == g["accepted_A"]
    assert r.overflow == g["dropped"]
    assert (r.accepted[0] <= r.C).all()


def test_overflow_token_keeps_its_raw_expert():
    # [070, 官方代码阅读路线]: re-taking argmax of a zeroed mask row returns 0;
    # the reported expert of an overflow token must stay its raw choice.
    T, E = 12, 4
    x = np.zeros((T, E))
    x[:, 2] = 1.0
    r = so.route(x, 3.0 * np.eye(E), None, 1, T, E, 1.0)  # C = 3
    assert r.C == 3
    assert (r.expert == 2).all()
    assert r.keep.sum() == 3 and (r.row[~r.keep] == -1).all()
    assert r.raw[0].tolist() == [0, 0, 12, 0] and r.accepted[0].tolist() == [0, 0, 3, 0]


# ----------------------------------------------------------------------------- ties and slots

def test_exact_ties_go_to_lowest_index():
    rng = np.random.default_rng(4)
    T, E, d = 40, 5, 6
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d))
    Wr[3] = Wr[1]          # experts 1 and 3 always tie exactly
    Wr[4] = Wr[0]          # experts 0 and 4 always tie exactly
    r = so.route(x, Wr, None, 1, T, E, 1.0)
    assert not np.isin(r.expert, [3, 4]).any()
    z = x @ Wr.T
    for t in range(T):
        assert r.expert[t] == min(np.flatnonzero(z[t] == z[t].max()))


def test_slots_match_cumulative_count_rule():
    rng = np.random.default_rng(5)
    for E in (1, 3, 17):
        a = rng.integers(0, E, size=300)
        for C in (0, 1, 5, 1000):
            slot, keep, raw, acc = so.assign_slots(a, E, C)
            np.testing.assert_array_equal(slot, cumsum_slots(a, E))
            np.testing.assert_array_equal(keep, cumsum_slots(a, E) < C)
            np.testing.assert_array_equal(raw, np.bincount(a, minlength=E))
            np.testing.assert_array_equal(acc, np.minimum(np.bincount(a, minlength=E), C))


def test_row_layout_packs_groups_in_order():
    rng = np.random.default_rng(6)
    G, T, E, d = 3, 20, 4, 5
    x = rng.standard_normal((G * T, d))
    Wr = rng.standard_normal((E, d))
    r = so.route(x, Wr, None, G, T, E, 1.0)
    for e in range(E):
        kept = [t for t in range(G * T) if r.keep[t] and r.expert[t] == e]   # group, then sequence order
        assert [r.row[t] for t in kept] == list(range(len(kept)))
        assert r.expert_rows[e] == len(kept)


# ----------------------------------------------------------------------------- FFN and whole pipeline

def test_expert_ffn_matches_triple_loop():
    rng = np.random.default_rng(7)
    n, d, F = 3, 5, 7
    x = rng.standard_normal((n, d))
    W1 = rng.standard_normal((F, d))
    b1 = rng.standard_normal(F)
    W2 = rng.standard_normal((d, F))
    b2 = rng.standard_normal(d)
    o = so.expert_ffn(x, W1, b1, W2, b2)
    for i in range(n):
        h = [max(0.0, sum(W1[f, k] * x[i, k] for k in range(d)) + b1[f]) for f in range(F)]
        for j in range(d):
            ref = sum(W2[j, f] * h[f] for f in range(F)) + b2[j]
            assert abs(o[i, j] - ref) < 1e-12


def test_toy_expert_parameter_count(golden):
    g = golden("toy_expert.json")
    from gen import make_inputs
    inp = make_inputs(WORKLOADS["tiny-e16-fp32"], 1, expert_bias_std=0.1)
    per_expert = sum(inp[k][0].numel() for k in ("W1", "b1", "W2", "b2"))
    assert per_expert == g["params_per_expert"]
    assert tuple(inp["Wr"].shape) == (g["E"], g["d_model"])


@pytest.mark.parametrize("G,T,E,d,F,c,ties", [
    (1, 16, 4, 6, 5, 1.0, 0),
    (2, 24, 5, 4, 6, 0.6, 1),
    (3, 10, 3, 5, 4, 2.0, 1),
    (1, 9, 1, 3, 2, 1.0, 0),
])
def test_pipeline_matches_dense_einsum(G, T, E, d, F, c, ties):
    rng = np.random.default_rng(100 + G * T + E)
    x = rng.standard_normal((G * T, d))
    Wr = rng.standard_normal((E, d))
    if ties and E >= 2:
        Wr[1] = Wr[0]
    br = rng.standard_normal(E) * 0.1
    W1 = rng.standard_normal((E, F, d))
    b1 = rng.standard_normal((E, F))
    W2 = rng.standard_normal((E, d, F))
    b2 = rng.standard_normal((E, d))
    C = so.capacity(c, T, E)
    y_ref, D, xe_groups, a_ref, p_ref = dense_einsum_forward(x, Wr, br, W1, b1, W2, b2, G, T, E, C)
    r, y, _ = so.forward(x, Wr, br, W1, b1, W2, b2, G, T, E, c)
    assert r.C == C
    np.testing.assert_array_equal(r.expert, a_ref)
    np.testing.assert_allclose(r.probs, p_ref, rtol=1e-13)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    # dropped tokens: exactly zero expert output
    assert (y[~r.keep] == 0).all()
    # dispatch buffer: each expert's block is its kept rows group by group, then zeros
    xe = so.dispatch(x, r, E, G)
    for e in range(E):
        blocks = [xe_groups[g, e, :r.accepted[g, e]] for g in range(G)]
        packed = np.concatenate(blocks, axis=0) if blocks else np.zeros((0, d))
        n = packed.shape[0]
        np.testing.assert_array_equal(xe[e, :n], packed)
        assert (xe[e, n:] == 0).all()
    # statistics from the one-hot tensor
    for g in range(G):
        np.testing.assert_array_equal(r.accepted[g], D[g].sum(axis=(0, 2)).astype(int))
    np.testing.assert_allclose(r.aux_per_group, 0.01 * r.balance)
    assert abs(r.aux_loss - np.mean(r.aux_per_group)) < 1e-15


def test_near_tie_detection():
    z = np.array([[1.0, 1.0 + 5e-7, 0.0], [0.0, 1.0, 2.0]])
    assert so.ties_within(z, 1e-6).tolist() == [True, False]
    assert so.groups_with_near_ties([z], G=2, T=1) == [0]


def test_choice_logits_decide_only_the_choices():
    # Substituted scores move group 1's tokens to expert 2; probabilities, gates and P stay
    # the float64 ones, and f (hence the balance term) follows the new choices.
    rng = np.random.default_rng(8)
    G, T, E, d = 2, 6, 3, 4
    x = rng.standard_normal((G * T, d))
    Wr = rng.standard_normal((E, d))
    z_alt = np.zeros((T, E))
    z_alt[:, 2] = 1.0
    r = so.route(x, Wr, None, G, T, E, 1.0, choice_logits={1: z_alt})
    r0 = so.route(x, Wr, None, G, T, E, 1.0)
    assert (r.expert[T:] == 2).all()
    np.testing.assert_array_equal(r.expert[:T], r0.expert[:T])
    np.testing.assert_array_equal(r.logits, r0.logits)
    np.testing.assert_array_equal(r.probs, r0.probs)
    np.testing.assert_array_equal(r.P, r0.P)
    assert r.z_loss == r0.z_loss
    np.testing.assert_array_equal(r.gate, r0.probs[np.arange(G * T), r.expert])
    np.testing.assert_array_equal(r.raw[1], [0, 0, T])
    assert r.balance[1] == E * r0.P[1][2]  # f = (0, 0, 1)
    np.testing.assert_array_equal(r.balance[0], r0.balance[0])
    # top-2: the substituted scores pick the pair; the gates come from the float64 scores
    z_alt2 = np.zeros((T, E))
    z_alt2[:, 2], z_alt2[:, 0] = 2.0, 1.0
    r2 = so.route_top2(x, Wr, None, G, T, E, 1.0, choice_logits={1: z_alt2})
    assert (r2.expert[T:] == 2).all() and (r2.expert2[T:] == 0).all()
    z = r0.logits[T:]
    np.testing.assert_allclose(r2.gate[T:], np.exp(z[:, 2]) / (np.exp(z[:, 2]) + np.exp(z[:, 0])), rtol=1e-14)


# ----------------------------------------------------------------------------- router z-loss

def test_z_loss_equal_scores_closed_form():
    # every score of a token equal to s_t: log sum_i e^{s_t} = s_t + ln E exactly
    for E in (1, 2, 7, 128, 2048):
        T = 5
        x = np.array([[0.0], [1.5], [-2.0], [0.25], [3.0]])
        Wr = np.ones((E, 1))
        r = so.route(x, Wr, None, 1, T, E, 1.0)
        want = float(np.mean((x[:, 0] + math.log(E)) ** 2))
        assert abs(r.z_loss - want) <= 1e-12 * max(1.0, want)
        # all-zero scores: (ln E)^2
        r0 = so.route(np.zeros((T, 1)), Wr, None, 1, T, E, 1.0)
        assert abs(r0.z_loss - math.log(E) ** 2) <= 1e-12 * max(1.0, math.log(E) ** 2)


def test_z_loss_dominant_score():
    # one score L far above the rest (zeros): log sum = L + log(1 + (E-1) e^-L) -> L^2 to 1e-12
    E, L = 64, 60.0
    br = np.zeros(E)
    br[5] = L
    r = so.route(np.zeros((3, 1)), np.zeros((E, 1)), br, 1, 3, E, 1.0)
    assert abs(r.z_loss - L * L) <= 1e-12 * L * L


def test_z_loss_changes_under_shift_but_routing_does_not(golden):
    g = golden("z_loss_shift.json")
    c = g["shift"]
    rng = np.random.default_rng(5)
    T, E, d = 40, 8, 6
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d)) * 0.3
    br = rng.standard_normal(E) * 0.1
    r0, r1, r2 = (so.route(x, Wr, br + k * c, 1, T, E, 1.0) for k in (0, 1, 2))
    assert (r1.expert == r0.expert).all() and (r1.slot == r0.slot).all()
    assert abs(r1.z_loss - r0.z_loss) > 1.0
    # (log sum exp(z + c))^2 = (lse + c)^2: quadratic in c with unit leading coefficient,
    # so the second difference over steps of c is exactly 2 c^2
    second = r2.z_loss - 2.0 * r1.z_loss + r0.z_loss
    assert abs(second - 2.0 * c * c) <= 1e-9 * c * c


def test_z_loss_is_per_group_then_mean():
    # two groups, every score of a token equal to x_t: group g's loss is mean_t (x_t + ln E)^2
    E, T = 4, 3
    x = np.array([[0.0], [0.0], [0.0], [2.0], [2.0], [2.0]])
    r = so.route(x, np.ones((E, 1)), None, 2, T, E, 1.0)
    lnE = math.log(E)
    np.testing.assert_allclose(r.z_per_group, [lnE ** 2, (2.0 + lnE) ** 2], rtol=1e-13)
    assert abs(r.z_loss - 0.5 * (lnE ** 2 + (2.0 + lnE) ** 2)) <= 1e-13 * r.z_loss


# ----------------------------------------------------------------------------- top-2 variant

def queue_top2_slots(a1, a2, E, C):
    """Second formulation of the top-2 slot rule: one queue of (token, choice) requests, all
    first choices in sequence order, then all second choices in sequence order; each expert
    accepts requests while it has fewer than C."""
    T = len(a1)
    taken = [0] * E
    slot = {}  # (token, choice) -> slot of an accepted request; None when refused
    for choice, a in ((0, a1), (1, a2)):
        for t in range(T):
            e = int(a[t])
            if taken[e] < C:
                slot[(t, choice)] = taken[e]
                taken[e] += 1
            else:
                slot[(t, choice)] = None
    return slot


def test_top2_gates_page_rule(golden):
    g = golden("top2_gates.json")
    E, d, T = g["E"], g["d"], 40
    rng = np.random.default_rng(3)
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d)) * math.sqrt(0.1 / d)
    r = so.route_top2(x, Wr, None, 1, T, E, 1.0)
    np.testing.assert_allclose(r.gate + r.gate2, g["weights_sum"], rtol=0, atol=1e-15)
    for t in range(T):
        z1, z2 = r.logits[t, r.expert[t]], r.logits[t, r.expert2[t]]
        assert z1 >= z2 and r.expert[t] != r.expert2[t]
        # softmax over the two kept scores: the first weight is the logistic of their gap
        assert abs(r.gate[t] - 1.0 / (1.0 + math.exp(-(z1 - z2)))) < 1e-15
        # and the two are the largest scores of the row
        assert (np.sort(r.logits[t])[-2:] == np.sort([z1, z2])).all()


def test_top2_two_experts_and_ties():
    # E = 2: both experts chosen; equal scores: experts 0 then 1, weights 1/2 each
    x = np.array([[0.7], [-1.2], [0.0]])
    Wr = np.array([[1.0], [0.0]])
    r = so.route_top2(x, Wr, None, 1, 3, 2, 1.0)
    assert r.expert.tolist() == [0, 1, 0] and r.expert2.tolist() == [1, 0, 1]
    assert abs(r.gate[2] - 0.5) < 1e-15 and abs(r.gate2[2] - 0.5) < 1e-15
    r4 = so.route_top2(np.zeros((5, 1)), np.ones((4, 1)), None, 1, 5, 4, 1.0)
    assert (r4.expert == 0).all() and (r4.expert2 == 1).all()


def test_top2_capacity_is_twice_top1():
    for (c, T, E) in [(1.0, 64, 4), (1.25, 4096, 64), (1.0, 8192, 128), (1.0, 32, 16)]:
        assert so.capacity(2 * c, T, E) == 2 * so.capacity(c, T, E)  # c T / E integral here
    r = so.route_top2(np.zeros((64, 1)), np.ones((4, 1)), None, 1, 64, 4, 1.0)
    assert r.C == 32


def test_top2_slots_match_queue_rule():
    rng = np.random.default_rng(9)
    for (G, T, E, c) in [(1, 30, 4, 0.5), (3, 17, 5, 1.0), (2, 40, 3, 0.25)]:
        x = rng.standard_normal((G * T, 3))
        Wr = rng.standard_normal((E, 3))
        br = np.array([0.8] + [0.0] * (E - 1))  # crowd expert 0
        r = so.route_top2(x, Wr, br, G, T, E, c)
        before = np.zeros(E, dtype=np.int64)
        for g in range(G):
            sl = slice(g * T, (g + 1) * T)
            q = queue_top2_slots(r.expert[sl], r.expert2[sl], E, r.C)
            for t in range(T):
                tt = g * T + t
                for (sl_, kp, rw, ex, ch) in ((r.slot, r.keep, r.row, r.expert, 0),
                                              (r.slot2, r.keep2, r.row2, r.expert2, 1)):
                    qs = q[(t, ch)]
                    assert bool(kp[tt]) == (qs is not None)
                    if qs is None:
                        assert sl_[tt] >= r.C and rw[tt] == -1
                    else:
                        assert sl_[tt] == qs and rw[tt] == before[ex[tt]] + qs
            kept = np.bincount(r.expert[sl][r.keep[sl]], minlength=E) + \
                np.bincount(r.expert2[sl][r.keep2[sl]], minlength=E)
            assert (kept <= r.C).all()
            assert (kept == r.accepted[g] + r.accepted2[g]).all()
            before += kept
        assert (r.expert_rows == before).all()
        # f counts first choices only, over all T tokens
        np.testing.assert_allclose(r.f.sum(axis=1), 1.0, rtol=1e-15)


def test_top2_without_drops_is_the_dense_weighted_pair():
    # enough capacity for every request: y_t = w1 FFN_e1(x_t) + w2 FFN_e2(x_t), computed here
    # densely (every expert on every token) with the pair found by a stable sort
    rng = np.random.default_rng(4)
    G, T, E, d, F = 2, 9, 5, 6, 7
    x = rng.standard_normal((G * T, d))
    Wr = rng.standard_normal((E, d))
    W1 = rng.standard_normal((E, F, d)) * 0.3
    b1 = rng.standard_normal((E, F)) * 0.1
    W2 = rng.standard_normal((E, d, F)) * 0.3
    b2 = rng.standard_normal((E, d)) * 0.1
    y, r = so.forward_top2(x, Wr, None, W1, b1, W2, b2, G, T, E, 1.0, capacity_override=2 * T)
    assert r.keep.all() and r.keep2.all()
    z = x @ Wr.T
    h = np.maximum(np.einsum("nd,efd->nef", x, W1) + b1[None], 0.0)
    o = np.einsum("nef,edf->ned", h, W2) + b2[None]
    order = np.argsort(-z, axis=1, kind="stable")
    want = np.zeros((G * T, d))
    for t in range(G * T):
        e1, e2 = order[t, 0], order[t, 1]
        w = np.exp(z[t, [e1, e2]] - z[t, e1])
        w = w / w.sum()
        want[t] = w[0] * o[t, e1] + w[1] * o[t, e2]
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- backward

def _loss(x, Wr, br, W1, b1, W2, b2, G, T, E, c, dy, w_aux, w_z, residual, fixed):
    """L = sum(dy * y) + w_aux aux + w_z z for the given parameters, from the oracle's
    forward pieces; `fixed` (expert, keep) must not change under the perturbation."""
    r = so.route(x, Wr, br, G, T, E, c)
    assert (r.expert == fixed[0]).all() and (r.keep == fixed[1]).all(), "a choice flipped"
    outs = so.expert_outputs(x, r, W1, b1, W2, b2)
    y = so.combine(r, outs, range(G * T), x.shape[1])
    if residual:
        y = y + x
    return float(np.sum(dy * y)) + w_aux * r.aux_loss + w_z * r.z_loss


@pytest.mark.parametrize("G,T,E,c,residual", [(1, 7, 3, 1.0, False), (2, 6, 4, 0.75, True)])
def test_backward_matches_central_differences(G, T, E, c, residual):
    # the pages' check: central differences over every parameter, routing unchanged by the step
    rng = np.random.default_rng(17)
    d, F = 4, 5
    x = rng.standard_normal((G * T, d))
    Wr = rng.standard_normal((E, d))
    br = rng.standard_normal(E) * 0.3
    W1 = rng.standard_normal((E, F, d))
    b1 = rng.standard_normal((E, F)) * 0.3
    W2 = rng.standard_normal((E, d, F))
    b2 = rng.standard_normal((E, d)) * 0.3
    dy = rng.standard_normal((G * T, d))
    w_aux, w_z = 0.7, 0.3
    grads = so.backward(x, Wr, br, W1, b1, W2, b2, G, T, E, c, dy, w_aux, w_z, residual=residual)
    r = grads["route"]
    assert (~r.keep).any() or c >= 1.0
    fixed = (r.expert.copy(), r.keep.copy())
    params = dict(x=x, Wr=Wr, br=br, W1=W1, b1=b1, W2=W2, b2=b2)
    eps = 1e-6
    worst = 0.0
    for name, arr in params.items():
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = arr[i]
            arr[i] = old + eps
            lp = _loss(**params, G=G, T=T, E=E, c=c, dy=dy, w_aux=w_aux, w_z=w_z, residual=residual, fixed=fixed)
            arr[i] = old - eps
            lm = _loss(**params, G=G, T=T, E=E, c=c, dy=dy, w_aux=w_aux, w_z=w_z, residual=residual, fixed=fixed)
            arr[i] = old
            num[i] = (lp - lm) / (2 * eps)
        ana = grads["d" + name]
        err = np.max(np.abs(ana - num))
        worst = max(worst, err)
        assert err < 1e-6 * max(1.0, np.max(np.abs(num))), f"d{name}: max |analytic - central difference| {err:.3e}"
    assert worst < 1e-6


def test_backward_gate_path_only_reaches_the_chosen_expert():
    # with w_aux = w_z = 0 the router gradient of a token is p_t * (e_a - p_t) * dg_t: rows sum to 0
    rng = np.random.default_rng(2)
    T, E, d, F = 9, 4, 3, 2
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d))
    W1 = rng.standard_normal((E, F, d))
    W2 = rng.standard_normal((E, d, F))
    dy = rng.standard_normal((T, d))
    g = so.backward(x, Wr, None, W1, None, W2, None, 1, T, E, 1.0, dy)
    # softmax Jacobian rows sum to zero, so dbr sums to zero
    assert abs(g["dbr"].sum()) < 1e-12
    # experts nobody kept get no weight gradient
    r = g["route"]
    for e in range(E):
        if not (r.keep & (r.expert == e)).any():
            assert (g["dW1"][e] == 0).all() and (g["dW2"][e] == 0).all()


# ----------------------------------------------------------------------------- expert parallelism

@pytest.mark.parametrize("world,E", [(2, 8), (3, 7), (4, 4)])
def test_sharded_experts_equal_the_single_rank_layer(world, E):
    # [card, 方法适配]: experts sharded over cores with two all-to-alls compute the same layer
    # as one core holding every expert over all the cores' routing groups: routing is per
    # group and each expert output depends on its own token only.  Uneven expert ranges
    # (E = 7 over 3 ranks) and one expert per rank are included.
    rng = np.random.default_rng(41 + world)
    G, T, d, F = 2, 24, 12, 10
    xs = [rng.standard_normal((G * T, d)) for _ in range(world)]
    Wr = rng.standard_normal((E, d)) * 0.4
    br = rng.standard_normal(E) * 0.2
    W1 = rng.standard_normal((E, F, d)) * 0.3
    b1 = rng.standard_normal((E, F)) * 0.1
    W2 = rng.standard_normal((E, d, F)) * 0.3
    b2 = rng.standard_normal((E, d)) * 0.1
    routes, ys = so.ep_forward(xs, Wr, br, W1, b1, W2, b2, G, T, E, 0.75, world)
    ref, y_ref, _ = so.forward(np.concatenate(xs), Wr, br, W1, b1, W2, b2, world * G, T, E, 0.75)
    N = G * T
    for r in range(world):
        sl = slice(r * N, (r + 1) * N)
        for f in ("expert", "slot", "keep", "gate"):
            np.testing.assert_array_equal(getattr(routes[r], f), getattr(ref, f)[sl], err_msg=f)
        np.testing.assert_allclose(routes[r].raw, ref.raw[r * G:(r + 1) * G])
        np.testing.assert_allclose(ys[r], y_ref[sl], rtol=1e-12, atol=1e-14)
    assert (~ref.keep).any() and ref.keep.any()  # c = 0.75 drops tokens
