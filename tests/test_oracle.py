"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself:
exact rational arithmetic, library routines (numpy matmul, lexsort, scipy
softmax), brute-force enumeration, closed forms from the pages' equations,
worked examples under tests/golden/, and stated invariants.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (test-side helper)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def rand_bf16(shape, scale=1.0, mean=0.0):
    return f32_to_bf16_bits((mean + scale * rng.standard_normal(shape)).astype(np.float32))


def widen(bits):
    return orc.bf16_to_f64(bits)


def exact_bf16(v: float) -> int:
    b = int(f32_to_bf16_bits(np.array([v], np.float32))[0])
    assert float(widen(np.array([b], np.uint16))[0]) == v, v
    return b


# ---------------------------------------------------------------- widening
def test_bf16_widening_is_exact():
    # IEEE binary32 upper halves: 1.0, -2.0, 0.5, largest finite, smallest subnormal
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x7F7F: 3.3895313892515355e38,
             0x0001: 2.0 ** -133, 0x0000: 0.0}
    lib = orc.lib()
    for b, v in cases.items():
        assert lib.orc_bf16_to_f64(b) == v


# ------------------------------------------------------------------ scores
def test_scores_match_exact_rational_dot():
    """bf16 products have <= 16 significant bits; with a bounded exponent spread
    the fp64 sum of 128 of them is exact, so z must equal the rational dot."""
    d, L = 128, 7
    q = rand_bf16(d)
    k = rand_bf16((L, d), 1.5, 0.25)
    z = orc.scores(q, k, 1.0)
    qf, kf = widen(q), widen(k)
    for i in range(L):
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qf, kf[i]))
        assert z[i] == float(exact)
    # the logit scale of Eq. 1 multiplies
    s = 1.0 / math.sqrt(d)
    zs = orc.scores(q, k, s)
    assert np.all(zs == s * z)


def test_scores_match_numpy_matmul():
    d, L = 128, 300
    q = rand_bf16(d)
    k = rand_bf16((L, d), 1.0, 0.3)
    z = orc.scores(q, k, 0.125)
    ref = 0.125 * (widen(k) @ widen(q))
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------- top-K
def brute_topk(z, pool, K):
    """Enumerate all K-subsets and keep the one that dominates every outsider
    under the order (z desc, index asc)."""
    pool = list(pool)
    K = min(K, len(pool))
    best = None
    for S in itertools.combinations(pool, K):
        Sset = set(S)
        ok = all((z[i] > z[j]) or (z[i] == z[j] and i < j)
                 for i in Sset for j in pool if j not in Sset)
        if ok:
            assert best is None, "two dominating sets"
            best = Sset
    return best


@pytest.mark.parametrize("trial", range(6))
def test_topk_bruteforce_tiny(trial):
    n = 9
    z = rng.integers(-3, 4, size=12).astype(np.float64)  # many exact ties
    pool = sorted(rng.choice(12, size=n, replace=False).tolist())
    for K in range(0, n + 2):
        got = orc.topk(z, pool, K)
        assert len(got) == min(K, n)
        assert set(got.tolist()) == (brute_topk(z, pool, K) if K > 0 else set())


def test_topk_matches_lexsort():
    n = 50_000
    z = np.round(rng.standard_normal(n), 3)  # ties are common after rounding
    pool = np.arange(n)
    K = 777
    got = orc.topk(z, pool, K)
    order = np.lexsort((pool, -z[pool]))
    assert np.array_equal(got, pool[order[:K]])


def test_topk_special_cases():
    z = rng.standard_normal(20)
    pool = np.arange(3, 17)
    assert len(orc.topk(z, pool, 0)) == 0
    assert sorted(orc.topk(z, pool, 14).tolist()) == pool.tolist()
    assert sorted(orc.topk(z, pool, 500).tolist()) == pool.tolist()


def test_topk_check_rules():
    z = np.array([5.0, 4.0, 3.0, 3.0 * (1 + 1e-9), 1.0, 0.5])
    pool = np.arange(6)
    # exact set for K=3 is {0, 1, 3}; positions 2 and 3 are a near-tie
    assert orc.topk_check(z, pool, 3, [3, 0, 1]) == 1
    assert orc.topk_check(z, pool, 3, [0, 1, 2]) == 2          # near-tie swap
    assert orc.topk_check(z, pool, 3, [0, 1, 4]) == 0          # far swap
    assert orc.topk_check(z, pool, 3, [0, 0, 1]) == 0          # duplicate
    assert orc.topk_check(z, pool, 3, [0, 1]) == 0             # wrong size
    assert orc.topk_check(z, pool[:5], 3, [0, 1, 5]) == 0      # outside pool
    assert orc.topk_check(z, pool, 0, []) == 1
    zt = np.array([5.0, 4.0, 3.0, 2.0])
    assert orc.topk_check(zt, np.arange(4), 2, [0, 2]) == 0    # gap 1.0: no tie


# ------------------------------------------------- partial attention, merge
def test_partial_closed_form():
    """Two keys with logits 0 and ln 3 get softmax weights 1/4 and 3/4."""
    z = np.array([0.0, math.log(3.0)])
    v = np.array([[exact_bf16(4.0), exact_bf16(-8.0)],
                  [exact_bf16(8.0), exact_bf16(16.0)]], np.uint16)
    o, m, l, lse = orc.partial(z, [0, 1], v)
    np.testing.assert_allclose(o, [0.25 * 4 + 0.75 * 8, 0.25 * -8 + 0.75 * 16], rtol=1e-15)
    assert m == math.log(3.0)
    assert abs(l - 4.0 / 3.0) < 1e-15
    assert abs(lse - math.log(4.0)) < 1e-15
    o, m, l, lse = orc.partial(z, [], v)
    assert np.all(o == 0) and lse == -math.inf and l == 0.0


def softmax_attend(z, idx, vf):
    from scipy.special import logsumexp, softmax
    idx = np.asarray(idx, np.int64)
    if len(idx) == 0:
        return np.zeros(vf.shape[1]), -math.inf
    w = softmax(z[idx])
    return w @ vf[idx], logsumexp(z[idx])


@pytest.mark.parametrize("trial", range(8))
def test_merge_of_disjoint_parts_equals_union(trial):
    """Eq. 4-5: the gamma rescale of two disjoint partials is softmax over the union."""
    L, d = 40, 16
    z = 6.0 * rng.standard_normal(L)
    v = rand_bf16((L, d))
    vf = widen(v)
    union = rng.choice(L, size=rng.integers(0, L), replace=False)
    cut = rng.integers(0, len(union) + 1)
    A, Bs = union[:cut], union[cut:]
    o1, m1, l1, _ = orc.partial(z, A, v)
    o2, m2, l2, _ = orc.partial(z, Bs, v)
    o, lse = orc.merge(o1, m1, l1, o2, m2, l2)
    ref, ref_lse = softmax_attend(z, union, vf)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    if len(union):
        assert abs(lse - ref_lse) < 1e-12
    else:
        assert lse == -math.inf


def test_merge_gamma_weights_literal():
    """gamma1 = e^(z1-z) l1 / (sum over the union) for a hand case."""
    o1, o2 = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    # W: logits {0, 0} -> m1 = 0, l1 = 2;  Omega: logits {ln 2} -> m2 = ln 2, l2 = 1
    o, lse = orc.merge(o1, 0.0, 2.0, o2, math.log(2.0), 1.0)
    # total mass 1 + 1 + 2 = 4: gamma1 = 2/4, gamma2 = 2/4
    np.testing.assert_allclose(o, [0.5, 0.5], rtol=1e-15)
    assert abs(lse - math.log(4.0)) < 1e-15


# ---------------------------------------------------------------- window
def test_window_ranges():
    def W(L, ni, nr):
        return [i for i in range(L) if orc.in_window(i, L, ni, nr)]
    assert W(10, 2, 3) == [0, 1, 7, 8, 9]
    assert W(4, 2, 3) == [0, 1, 2, 3]          # ranges overlap: union
    assert W(5, 0, 0) == []
    assert W(5, 0, 2) == [3, 4]
    assert W(5, 7, 0) == [0, 1, 2, 3, 4]       # clipped to the cache
    assert W(0, 3, 3) == []


# ------------------------------------------------------- whole decode step
def test_worked_example_golden():
    rows = [l.split() for l in open(os.path.join(GOLD, "attention_worked_example.txt"))
            if l.strip() and not l.startswith("#")]
    k = np.array([[exact_bf16(float(r[1])), exact_bf16(float(r[2]))] for r in rows], np.uint16)
    v = np.array([[exact_bf16(float(r[3])), exact_bf16(float(r[4]))] for r in rows], np.uint16)
    q = np.array([exact_bf16(1.0), exact_bf16(0.0)], np.uint16)
    r = orc.decode_head(q, k, v, K=2, n_init=1, n_recent=1, scale=1.0)
    e2, e3 = math.exp(2), math.exp(3)
    den = 2 + e3 + e2
    assert sorted(r["sel"].tolist()) == [1, 2]
    np.testing.assert_allclose(r["out"], [(1 + 2 * e3) / den, (8 + 2 * e3 + e2) / den],
                               rtol=1e-14)
    assert abs(r["lse"] - math.log(den)) < 1e-14


def _decode_inputs(L, d=128, plant=5):
    q = rand_bf16(d)
    k = rand_bf16((L, d), 1.0, 0.2)
    pos = rng.choice(L, size=plant, replace=False)
    k[pos] = f32_to_bf16_bits(0.05 * widen(q)[None, :] + 0.1 * rng.standard_normal((plant, d)))
    v = rand_bf16((L, d))
    return q, k, v


@pytest.mark.parametrize("L,ni,nr", [(300, 4, 16), (50, 30, 30), (257, 0, 0), (1, 1, 1)])
def test_K_covering_pool_equals_full_softmax(L, ni, nr):
    """K >= |P|: W u Omega = [0, L), so the step is full softmax attention (Eq. 1)."""
    q, k, v = _decode_inputs(L, plant=1)
    s = 1 / math.sqrt(128)
    r = orc.decode_head(q, k, v, K=L, n_init=ni, n_recent=nr, scale=s)
    zf = s * (widen(k) @ widen(q))
    ref, ref_lse = softmax_attend(zf, np.arange(L), widen(v))
    np.testing.assert_allclose(r["out"], ref, rtol=1e-11, atol=1e-12)
    assert abs(r["lse"] - ref_lse) < 1e-11


def test_K0_is_window_only_attention():
    """K = 0: only the static pattern is attended (the StreamingLLM case)."""
    L, ni, nr = 400, 4, 32
    q, k, v = _decode_inputs(L)
    s = 1 / math.sqrt(128)
    r = orc.decode_head(q, k, v, K=0, n_init=ni, n_recent=nr, scale=s)
    zf = s * (widen(k) @ widen(q))
    win = list(range(ni)) + list(range(L - nr, L))
    ref, ref_lse = softmax_attend(zf, win, widen(v))
    np.testing.assert_allclose(r["out"], ref, rtol=1e-11, atol=1e-12)
    assert len(r["sel"]) == 0


def test_selection_is_disjoint_from_window_and_exact():
    L, ni, nr, K = 1000, 8, 64, 50
    q, k, v = _decode_inputs(L, plant=20)
    s = 1 / math.sqrt(128)
    r = orc.decode_head(q, k, v, K=K, n_init=ni, n_recent=nr, scale=s)
    sel = set(r["sel"].tolist())
    assert not sel & (set(range(ni)) | set(range(L - nr, L)))
    zf = s * (widen(k) @ widen(q))
    pool = np.array([i for i in range(L) if not (i < ni or i >= L - nr)])
    order = np.lexsort((pool, -zf[pool]))
    assert sel == set(pool[order[:K]].tolist())
    ref, _ = softmax_attend(zf, sorted(sel | set(range(ni)) | set(range(L - nr, L))), widen(v))
    np.testing.assert_allclose(r["out"], ref, rtol=1e-11, atol=1e-12)
