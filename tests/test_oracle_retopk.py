"""Pins of the ReTopK oracle ("Recall Before You Rank", method sections 1-5).

Checked against stated invariants (M_t <= RK+W, the recent window is always
a candidate, candidates come only from recalled supports), special cases that
reduce to exact top-K (T_r = 1, tau > 1), the W = 0 failure mechanism, the
exact-recovery property, the strict fallback, the FIFO discipline and the
page's worked bound 2080 (tests/golden/retopk_candidate_bound.txt).  Exact
top-K references use numpy (matmul + lexsort), not the oracle.
"""
import math
import os

import numpy as np
import pytest

import oracle as orc
from test_oracle import f32_to_bf16_bits, widen

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(777)
D = 128


def np_topk(q, k, L, K):
    z = widen(k[:L]) @ widen(q)
    pool = np.arange(L)
    order = np.lexsort((pool, -z))
    return set(pool[order[:K]].tolist())


def make_case(L_total=400, Hq=1, walk_rho=0.97, steps=12):
    k = f32_to_bf16_bits(0.3 + rng.standard_normal((L_total, D)))
    v = f32_to_bf16_bits(rng.standard_normal((L_total, D)))
    qs = []
    qb = rng.standard_normal((Hq, D))
    qb /= np.linalg.norm(qb, axis=1, keepdims=True)
    for _ in range(steps + 8):
        qb = walk_rho * qb + math.sqrt(1 - walk_rho ** 2) * rng.standard_normal((Hq, D)) / math.sqrt(D)
        qb /= np.linalg.norm(qb, axis=1, keepdims=True)
        qs.append(f32_to_bf16_bits(qb * math.sqrt(D)))
    return k, v, qs


def init_from_prefill(st, k, qs_pre, L0, K):
    """Slot c <- prefill query at position L0-C+c with its exact causal top-K."""
    Cn = len(qs_pre)
    for c in range(Cn):
        p = L0 - Cn + c
        for h in range(st.Hq):
            st.set_slot(h, c, qs_pre[c][h], sorted(np_topk(qs_pre[c][h], k, p + 1, K)))


def run(st, k, v, qs, L0, steps, check=None):
    out = []
    for t in range(steps):
        L = L0 + t + 1
        for h in range(st.Hq):
            before = [st.slot_support(h, c) for c in range(st.C)]
            r = st.step_head(h, qs[t][h], k[:L], v[:L], 1 / math.sqrt(D))
            if check:
                check(t, h, L, r, before)
            out.append((t, h, r))
        st.advance()
    return out


def test_invariants_over_a_run():
    K, Cn, R, W, L0, steps = 16, 6, 2, 5, 300, 14
    k, v, qs = make_case(L0 + steps + 1, Hq=2, steps=steps)
    st = orc.ReTopK(2, D, K, Cn, R, W, tau=0.2, T_r=6)
    init_from_prefill(st, k, qs[:Cn], L0, K)

    def check(t, h, L, r, before):
        if r["path"] == 1:
            assert t % 6 == 0 or r["max_rho"] < 0.2
            assert set(r["sup"].tolist()) == np_topk(qs[Cn + t][h], k, L, K)
            return
        A = r["cand"]
        assert len(A) <= R * K + W                        # M_t <= RK + W
        assert np.all(np.diff(A) > 0)                     # unique, ascending
        assert set(range(L - W, L)) <= set(A.tolist())    # recent window kept
        pooled = set().union(*[set(b.tolist()) for b in before]) | set(range(L - W, L))
        assert set(A.tolist()) <= pooled                  # only recalled supports
        assert set(r["sup"].tolist()) <= set(A.tolist())
        assert len(r["sup"]) == min(K, len(A))
        # re-top-K over A by the current query's exact scores
        zA = widen(k[A]) @ widen(qs[Cn + t][h])
        order = np.lexsort((A, -zA))
        assert set(r["sup"].tolist()) == set(A[order[:K]].tolist())

    shifted = qs[Cn:]
    res = run(st, k, v, shifted, L0, steps, check)
    paths = [r["path"] for _, _, r in res]
    assert 0 in paths and 1 in paths


def test_refresh_every_step_is_exact_topk():
    K, Cn, R, W, L0, steps = 12, 4, 2, 3, 250, 6
    k, v, qs = make_case(L0 + steps + 1, steps=steps)
    for tau, T_r in [(0.0, 1), (1.5, 1000)]:   # T_r = 1, or tau > 1
        st = orc.ReTopK(1, D, K, Cn, R, W, tau=tau, T_r=T_r)
        init_from_prefill(st, k, qs[:Cn], L0, K)
        for t, h, r in run(st, k, v, qs[Cn:], L0, steps):
            assert r["path"] == 1
            assert set(r["sup"].tolist()) == np_topk(qs[Cn + t][h], k, L0 + t + 1, K)


def test_no_fallback_reuses_after_step0():
    K, Cn, R, W, L0, steps = 12, 4, 2, 3, 250, 8
    k, v, qs = make_case(L0 + steps + 1, steps=steps, walk_rho=0.5)
    st = orc.ReTopK(1, D, K, Cn, R, W, tau=-1.5, T_r=10_000)
    init_from_prefill(st, k, qs[:Cn], L0, K)
    paths = [r["path"] for _, _, r in run(st, k, v, qs[Cn:], L0, steps)]
    assert paths == [1] + [0] * (steps - 1)


def test_W0_never_admits_fresh_tokens():
    """ReTopK section 3: without the recent window a token appended after the
    last exact step can never enter a candidate set."""
    K, Cn, R, L0, steps = 10, 4, 2, 200, 10
    k, v, qs = make_case(L0 + steps + 1, steps=steps)
    # make every fresh token extremely attractive so exact top-K would take it
    for t in range(1, steps):
        k[L0 + t] = f32_to_bf16_bits(4.0 * widen(qs[Cn + t][0]))
    st = orc.ReTopK(1, D, K, Cn, R, 0, tau=-1.5, T_r=10_000)
    init_from_prefill(st, k, qs[:Cn], L0, K)
    for t, h, r in run(st, k, v, qs[Cn:], L0, steps):
        if t >= 1:
            assert r["path"] == 0
            assert max(r["sup"]) <= L0  # nothing appended at steps >= 1
    # with W >= 1 the newest token is always a candidate and, here, selected
    st = orc.ReTopK(1, D, K, Cn, R, 1, tau=-1.5, T_r=10_000)
    init_from_prefill(st, k, qs[:Cn], L0, K)
    for t, h, r in run(st, k, v, qs[Cn:], L0, steps):
        if t >= 1:
            assert (L0 + t) in r["cand"]
            assert (L0 + t) in r["sup"]


def test_exact_recovery_when_candidates_cover_topk():
    """If the exact S_t is inside A_t, re-ranking recovers exactly S_t."""
    K, Cn, R, W, L0 = 20, 4, 1, 2, 500
    k, v, qs = make_case(L0 + 3, steps=2)
    st = orc.ReTopK(1, D, K, Cn, R, W, tau=-1.5, T_r=10_000)
    q1 = qs[Cn + 1][0]
    S1 = sorted(np_topk(q1, k, L0 + 2, K))
    for c in range(Cn):  # every cached entry already holds step 1's answer
        st.set_slot(0, c, q1, S1)
    # step 0 (a refresh) uses an unrelated query, so its pushed entry is not recalled
    res = run(st, k, v, [[basis_query(5)], [q1]], L0, 2)
    r1 = res[1][2]
    assert r1["path"] == 0
    assert set(r1["sup"].tolist()) == set(S1)
    # output equals exact top-K softmax attention over S1 (no window)
    from scipy.special import softmax
    z = (widen(k[S1]) @ widen(q1)) / math.sqrt(D)
    np.testing.assert_allclose(r1["out"], softmax(z) @ widen(v[S1]), rtol=1e-11, atol=1e-12)


def basis_query(j):
    q = np.zeros(D, np.float32)
    q[j] = 2.0
    return f32_to_bf16_bits(q)


def test_fallback_is_strict_and_ties_prefer_older_slot():
    K, Cn, R, W, L0 = 4, 3, 1, 1, 100
    k, v, _ = make_case(L0 + 4, steps=2)
    e0, e1 = basis_query(0), basis_query(1)
    supp = [[10, 11, 12, 13], [20, 21, 22, 23], [30, 31, 32, 33]]
    for tau, want_path in [(1.0, 0), (float(np.nextafter(1.0, 2.0)), 1)]:
        st = orc.ReTopK(1, D, K, Cn, R, W, tau=tau, T_r=10_000)
        st.set_slot(0, 0, e1, supp[0])
        st.set_slot(0, 1, e0, supp[1])   # older of the two exact matches
        st.set_slot(0, 2, e0, supp[2])
        run(st, k, v, [[e1]], L0, 1)     # step 0 (refresh) evicts slot 0
        r = st.step_head(0, e0, k[:L0 + 2], v[:L0 + 2], 1 / math.sqrt(D))
        assert r["max_rho"] == 1.0
        assert r["path"] == want_path    # max rho == tau -> reuse
        if want_path == 0:
            assert r["cand"].tolist() == supp[1] + [L0 + 1]


def test_fifo_push_on_both_paths_evicts_oldest():
    K, Cn, R, W, L0, steps = 6, 3, 1, 2, 150, 5
    k, v, qs = make_case(L0 + steps + 1, steps=steps)
    st = orc.ReTopK(1, D, K, Cn, R, W, tau=0.5, T_r=2)
    init_from_prefill(st, k, qs[:Cn], L0, K)
    for t in range(steps):
        ages = [st.slot_age(0, c) for c in range(Cn)]
        oldest = int(np.argmin(ages))
        r = st.step_head(0, qs[Cn + t][0], k[:L0 + t + 1], v[:L0 + t + 1], 1 / math.sqrt(D))
        assert sorted(st.slot_support(0, oldest).tolist()) == sorted(r["sup"].tolist())
        assert st.slot_age(0, oldest) == max(st.slot_age(0, c) for c in range(Cn))
        qb = widen(qs[Cn + t][0])
        np.testing.assert_allclose(st.slot_qbar(0, oldest), qb / np.linalg.norm(qb), rtol=1e-15)
        st.advance()


def test_candidate_bound_golden():
    """The page's bound: R=4, K=512, W=32 gives at most 2080 candidates, reached
    exactly when the recalled supports are disjoint and avoid the window."""
    rows = [l.split() for l in open(os.path.join(GOLD, "retopk_candidate_bound.txt"))
            if l.strip() and not l.startswith("#")]
    R, K, W, bound = map(int, rows[0])
    assert R * K + W == bound
    Cn, L0 = R + 1, 3000
    k, v, _ = make_case(L0 + 3, steps=1)
    e0, e1 = basis_query(0), basis_query(1)
    st = orc.ReTopK(1, D, K, Cn, R, W, tau=-1.5, T_r=10_000)
    st.set_slot(0, 0, e1, list(range(0, K)))           # evicted by step 0
    for c in range(1, Cn):
        st.set_slot(0, c, e0, list(range(c * K - K, c * K)))  # disjoint blocks
    run(st, k, v, [[e1]], L0, 1)
    r = st.step_head(0, e0, k[:L0 + 2], v[:L0 + 2], 1 / math.sqrt(D))
    assert r["path"] == 0
    assert r["n_cand"] == bound


# ---------------------------------------------------------------------------
# Lockstep adoption.  The parity tests run the oracle beside the GPU and let
# the oracle take the GPU's decision where its own lies within a rounding
# margin of a boundary (ReTopK "Fallback and refresh": max rho vs tau; the
# top-R recall at the R-th / (R+1)-th cosine; the exact top-K near-tie).  The
# cases below drive every such branch with cosines and logits that are known
# in closed form, inside and just outside each margin.
MARGIN = 1e-5  # the parity tests' path_abs / rho_abs


def vec(*pairs):
    """bf16 bits of the query with the given (channel, value) entries; every
    value used here is exact in bf16."""
    x = np.zeros(D, np.float32)
    for j, val in pairs:
        x[j] = val
    return f32_to_bf16_bits(x)


def tie_state(tau, R=2, T_r=10_000, margin=MARGIN):
    """Five slots against the step-1 query 2*e0 (closed-form cosines):
        slot 0: evicted by step 0 (a refresh step with query e5)
        slot 1: 2*e0                    rho = 1
        slot 2: e0 + 0.5 e1             rho = 1/sqrt(1.25)
        slot 3: e0 + 0.5 e1 + 2^-12 e2  rho = 1/sqrt(1.25 + 2^-24)  (2.1e-8 below slot 2)
        slot 4: e1                      rho = 0
    Supports are disjoint blocks, so every recalled set has its own union."""
    K, Cn, W, L0 = 4, 5, 2, 120
    k, v, _ = make_case(L0 + 3, steps=1)
    st = orc.ReTopK(1, D, K, Cn, R, W, tau=tau, T_r=T_r,
                    path_abs=margin, rho_abs=margin, topk_rel=1e-6)
    sup = {c: list(range(10 * c, 10 * c + K)) for c in range(Cn)}
    slots = [vec((5, 1.0)), vec((0, 2.0)), vec((0, 1.0), (1, 0.5)),
             vec((0, 1.0), (1, 0.5), (2, 2.0 ** -12)), vec((1, 1.0))]
    for c in range(Cn):
        st.set_slot(0, c, slots[c], sup[c])
    # step 0: refresh (t % T_r == 0), evicts slot 0 (the oldest)
    st.step_head(0, vec((5, 2.0)), k[:L0 + 1], v[:L0 + 1], 1 / math.sqrt(D))
    st.advance()
    L = L0 + 2
    recent = list(range(L - W, L))
    return st, k[:L], v[:L], sup, recent


def union(*parts):
    return sorted(set().union(*[set(p) for p in parts]))


def test_closed_form_cosines_of_the_tie_state():
    st, k, v, sup, recent = tie_state(tau=-1.5)
    r = st.step_head(0, vec((0, 2.0)), k, v, 1 / math.sqrt(D))
    assert r["max_rho"] == 1.0
    r2, r3 = 1 / math.sqrt(1.25), 1 / math.sqrt(1.25 + 2.0 ** -24)
    assert 0 < r2 - r3 < MARGIN
    # free run: R = 2 recalls slots 1 and 2 (slot 2's cosine is the larger of the tie)
    assert r["path"] == 0 and r["adopt_path"] == 0 and r["adopt_cand"] == 0
    assert r["cand"].tolist() == union(sup[1], sup[2], recent)


@pytest.mark.parametrize("offset,own,other,adopted", [
    (+0.5, 1, 0, True),    # own exact (1 < tau), inside the margin: take the other's reuse
    (+2.0, 1, 0, False),   # just outside the margin: keep exact
    (-0.5, 0, 1, True),    # own reuse (1 >= tau), inside: take the other's exact path
    (-2.0, 0, 1, False),   # outside: keep reuse
])
def test_path_adoption_only_within_margin(offset, own, other, adopted):
    tau = 1.0 + offset * MARGIN
    st, k, v, sup, recent = tie_state(tau=tau)
    q = vec((0, 2.0))
    r = st.step_head(0, q, k, v, 1 / math.sqrt(D), other_path=other)
    assert r["own_path"] == own
    assert r["adopt_path"] == int(adopted)
    assert r["path"] == (other if adopted else own)
    if r["path"] == 1:  # exact path: the exact top-K of every key, no window
        assert set(r["sup"].tolist()) == np_topk(q, k, len(k), 4)
        assert r["n_cand"] == len(k)
    else:
        assert r["cand"].tolist() == union(sup[1], sup[2], recent)


def test_refresh_step_never_adopts_a_reuse_path():
    # step 1 with T_r = 1 is a refresh: max rho = 1 sits right at tau, the
    # other side claims reuse, the oracle stays exact
    st, k, v, sup, recent = tie_state(tau=1.0 - 0.5 * MARGIN, T_r=1)
    r = st.step_head(0, vec((0, 2.0)), k, v, 1 / math.sqrt(D), other_path=0)
    assert r["path"] == 1 and r["own_path"] == 1 and r["adopt_path"] == 0


@pytest.mark.parametrize("which,ok,adopt", [
    ("own", 1, 0),          # the same union: equal, nothing adopted
    ("tie_swap", 2, 1),     # the tied slot 3 instead of slot 2: an admissible choice
    ("drop_sure", 0, 0),    # both tied slots, the sure slot 1 dropped
    ("below_band", 0, 0),   # slot 4 (rho = 0) instead of a tied slot
    ("extra", 0, 0),        # the admissible union plus one stray position
])
def test_candidate_adoption_at_the_recall_boundary(which, ok, adopt):
    st, k, v, sup, recent = tie_state(tau=-1.5)
    other = {"own": union(sup[1], sup[2], recent),
             "tie_swap": union(sup[1], sup[3], recent),
             "drop_sure": union(sup[2], sup[3], recent),
             "below_band": union(sup[1], sup[4], recent),
             "extra": union(sup[1], sup[3], recent, [77])}[which]
    r = st.step_head(0, vec((0, 2.0)), k, v, 1 / math.sqrt(D), other_path=0,
                     other_cand=other)
    assert r["path"] == 0
    assert r["cand_ok"] == ok and r["adopt_cand"] == adopt
    if ok:  # the oracle continues with the other side's (admissible) union
        assert r["cand"].tolist() == other
    else:   # it keeps its own union, and the step counts as a mismatch
        assert r["cand"].tolist() == union(sup[1], sup[2], recent)


def test_candidate_adoption_needs_a_near_tie():
    # the same unions with margins far below the 2.1e-8 gap between slots 2
    # and 3: no tie at the boundary, so the swapped union is rejected
    st, k, v, sup, recent = tie_state(tau=-1.5, margin=1e-9)
    r = st.step_head(0, vec((0, 2.0)), k, v, 1 / math.sqrt(D), other_path=0,
                     other_cand=union(sup[1], sup[3], recent))
    assert r["cand_ok"] == 0 and r["adopt_cand"] == 0


@pytest.mark.parametrize("swap,ok", [(20, 2), (30, 0)])
def test_support_adoption_pushes_the_accepted_set(swap, ok):
    """Exact path (step 0 refresh), K = 3: positions 5 and 6 score 6s, 10 scores
    (2 + 2^-20)s and 20 scores 2s, every other key 0.  {5, 6, 20} differs from
    the exact {5, 6, 10} by a relative gap of 4.8e-7 < 1e-6 (accepted, and the
    FIFO receives it); {5, 6, 30} swaps in a key of logit 0 (rejected: the FIFO
    receives the oracle's own set)."""
    K, L = 3, 64
    k = np.zeros((L, D), np.float32)
    k[5, 0] = k[6, 0] = 3.0
    k[10, 0], k[10, 1] = 1.0, 1.0
    k[20, 0] = 1.0
    k = f32_to_bf16_bits(k)
    v = f32_to_bf16_bits(rng.standard_normal((L, D)))
    q = vec((0, 2.0), (1, 2.0 ** -20))
    st = orc.ReTopK(1, D, K, 2, 1, 2, tau=0.5, T_r=10_000,
                    path_abs=MARGIN, rho_abs=MARGIN, topk_rel=1e-6)
    st.set_slot(0, 0, vec((3, 1.0)), [1, 2, 3])
    st.set_slot(0, 1, vec((4, 1.0)), [1, 2, 3])
    other = [5, 6, swap]
    r = st.step_head(0, q, k, v, 1 / math.sqrt(D), other_path=1, other_sup=other)
    assert r["path"] == 1 and r["sup_ok"] == ok
    pushed = sorted(st.slot_support(0, 0).tolist())   # slot 0 was the oldest
    want = other if ok == 2 else [5, 6, 10]
    assert pushed == sorted(want) and sorted(r["sup"].tolist()) == sorted(want)
    # the output is the softmax over the pushed set
    from scipy.special import softmax
    z = (widen(k[want]) @ widen(q)) / math.sqrt(D)
    np.testing.assert_allclose(r["out"], softmax(z) @ widen(v[want]), rtol=1e-11, atol=1e-12)
