"""Pins of the oracle's acceptance rules, sampler, commit and draft-length schedule.

The rejection-sampling law is checked exactly: for a tiny vocabulary every
draft token is enumerated with its probability and every one of the 2^24
uniforms is accounted for by locating the points where the oracle's decision
changes (the decisions are monotone in the uniform), so the emitted token's
distribution is computed without Monte Carlo and compared with p within the
sampler's discretisation bound.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import accept as A
from oracle.analytic import expected_tokens_positional

TWO24 = 1 << 24


def _u(m):
    return np.float32(m * 2.0 ** -24)


def _first_true(pred, lo=0, hi=TWO24):
    """Smallest m in [lo, hi] with pred(m) true (pred monotone false->true); hi if none."""
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(mid):
            hi = mid
        else:
            lo = mid + 1
    return lo


def _sampler_law(w):
    """Exact law of ``A.sample_index(w, u)`` over all 2^24 uniforms (Fractions)."""
    V = len(w)
    law = [Fraction(0)] * V
    m = 0
    while m < TWO24:
        y = A.sample_index(w, _u(m))
        end = _first_true(lambda mm: A.sample_index(w, _u(mm)) != y, m, TWO24)
        law[y] += Fraction(end - m, TWO24)
        m = end
    return law


def _rand_rows(rng, V, n, sparse=False):
    z = rng.standard_normal((n, V)) * 1.5
    if sparse:
        z[:, rng.integers(0, V)] = -np.inf
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def test_sample_threshold_is_floor():
    rng = np.random.default_rng(0)
    for _ in range(2000):
        S = int(rng.integers(1, 1 << 47))
        m = int(rng.integers(0, TWO24))
        assert A.sample_threshold(S, m) == (m * S) >> 24


def test_sampler_law_matches_weights():
    w = np.array([5, 0, 1 << 30, 7, 1 << 29, 3], dtype=np.uint64)
    law = _sampler_law(w)
    S = int(w.sum())
    for y in range(len(w)):
        assert abs(float(law[y]) - int(w[y]) / S) <= 2.0 ** -24 + 1e-18
    assert law[1] == 0          # zero weight is never drawn


def test_sampler_picks_smallest_prefix_above_threshold():
    w = np.array([3, 0, 2, 5], dtype=np.uint64)   # prefix sums 3,3,5,10
    S = 10
    for m in (0, 1, TWO24 // 2, TWO24 - 1):
        t = (m * S) >> 24
        want = next(i for i, c in enumerate(np.cumsum(w)) if c > t)
        assert A.sample_index(w, _u(m)) == want


def test_int_weights_exact():
    r = np.array([0.0, 2.0 ** -32, 2.0 ** -33, 0.5, 1.0, 3 * 2.0 ** -20], dtype=np.float32)
    assert list(A.int_weights(r)) == [0, 1, 0, 1 << 31, 1 << 32, 3 << 12]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rejection_sampling_law_equals_target(seed):
    """Emitted first token ~ p and the bonus token ~ p[1] (k = 1, V = 5)."""
    rng = np.random.default_rng(seed)
    V = 5
    p = _rand_rows(rng, V, 2, sparse=(seed == 2))
    q = _rand_rows(rng, V, 1)
    first = [0.0] * V
    bonus_given_keep = {}
    for x in range(V):
        qx = float(q[0, x])
        if qx == 0.0:
            continue
        # uniforms u0 that keep x: the oracle's test is monotone (keep for small u0)
        keep_end = _first_true(lambda m: not A.ratio_accept(_u(m), q[0, x], p[0, x]))
        keep = keep_end / TWO24
        first[x] += qx * keep
        # on rejection, the residual draw is driven by u[1]: exact law over u[1]
        if keep_end < TWO24:
            m_rej = keep_end
            res_law = _sampler_law_of(lambda m: A.accept_sampling_chain(
                p, q, [x], [_u(m_rej), _u(m)])[1], V)
            assert A.accept_sampling_chain(p, q, [x], [_u(m_rej), _u(0)])[0] == 0
            for y in range(V):
                first[y] += qx * (1 - keep) * res_law[y]
        if keep_end > 0:
            bonus_given_keep[x] = _sampler_law_of(lambda m: A.accept_sampling_chain(
                p, q, [x], [_u(0), _u(m)])[1], V)
    tol = 4 * 2.0 ** -24 + V * 2.0 ** -30 + V * 2.0 ** -23
    np.testing.assert_allclose(first, p[0].astype(np.float64), rtol=0, atol=tol)
    for law in bonus_given_keep.values():
        np.testing.assert_allclose(law, p[1].astype(np.float64), rtol=0, atol=tol)


def _sampler_law_of(f, V):
    law = [0.0] * V
    m = 0
    while m < TWO24:
        y = f(m)
        end = _first_true(lambda mm: f(mm) != y, m, TWO24)
        law[y] += (end - m) / TWO24
        m = end
    return law


def test_acceptance_probability_is_overlap():
    """P(keep) = sum_x q(x) min(1, p(x)/q(x)) = sum_x min(p(x), q(x))."""
    rng = np.random.default_rng(7)
    V = 6
    p = _rand_rows(rng, V, 1)
    q = _rand_rows(rng, V, 1)
    pk = 0.0
    for x in range(V):
        keep_end = _first_true(lambda m: not A.ratio_accept(_u(m), q[0, x], p[0, x]))
        pk += float(q[0, x]) * keep_end / TWO24
    beta = float(np.minimum(p[0].astype(np.float64), q[0].astype(np.float64)).sum())
    assert abs(pk - beta) < V * 2.0 ** -24 + 1e-12


def test_zero_draft_probability_rejects():
    p = np.array([[0.5, 0.5, 0.0], [1 / 3, 1 / 3, 1 / 3]], dtype=np.float32)
    q = np.array([[0.0, 0.5, 0.5]], dtype=np.float32)
    a, nxt = A.accept_sampling_chain(p, q, [0], np.array([0.0, 0.0], dtype=np.float32))
    assert a == 0
    # residual max(0, p - q) = [0.5, 0, 0]: the correction must be token 0
    assert nxt == 0


def test_residual_all_zero_falls_back_to_p():
    # q(x) = 0 forces a rejection; with p == q elsewhere the residual is all zero,
    # so the correction is drawn from p itself (u = 0.125 -> token 0, u = 0.5 -> token 1)
    p = np.array([[0.25, 0.75, 0.0], [0.5, 0.5, 0.0]], dtype=np.float32)
    q = p[:1].copy()
    assert int(A.int_weights(A.residual(p[0], q[0])).sum()) == 0
    assert A.accept_sampling_chain(p, q, [2], np.array([0.0, 0.125], dtype=np.float32)) == (0, 0)
    assert A.accept_sampling_chain(p, q, [2], np.array([0.0, 0.5], dtype=np.float32)) == (0, 1)
    # p == q on a drawable token: always kept
    assert A.accept_sampling_chain(p, q, [1], np.array([1 - 2.0 ** -24, 0.5], dtype=np.float32))[0] == 1


def test_residual_is_clipped():
    p = np.array([0.1, 0.6, 0.3], dtype=np.float32)
    q = np.array([0.5, 0.2, 0.3], dtype=np.float32)
    r = A.residual(p, q)
    assert r[0] == 0 and r[2] == 0 and r[1] == np.float32(0.6) - np.float32(0.2)


def test_greedy_chain_bounds():
    V = 7
    logits = np.random.default_rng(3).standard_normal((5, V))
    am = logits.argmax(axis=1)
    a, nxt = A.accept_greedy_chain(am[:4], logits)      # every draft = target argmax
    assert a == 4 and nxt == am[4]                       # k+1 tokens emitted
    bad = am[:4].copy()
    bad[0] = (bad[0] + 1) % V
    a, nxt = A.accept_greedy_chain(bad, logits)
    assert a == 0 and nxt == am[0]                       # exactly one token emitted
    bad = am[:4].copy()
    bad[2] = (bad[2] + 1) % V
    assert A.accept_greedy_chain(bad, logits) == (2, am[2])


def test_argmax_ties_lowest():
    assert A.argmax_lowest([1.0, 3.0, 3.0, 2.0]) == 1


def _brute_tree(tokens, parents, logits):
    """Enumerate every node, check its whole root path, keep the deepest (lowest id)."""
    best = (0, 0)
    for i in range(len(tokens)):
        path = A.tree_path(parents, i)
        if all(tokens[path[d]] == int(np.argmax(logits[path[d - 1]])) for d in range(1, len(path))):
            cand = (len(path) - 1, -i)
            if cand > (best[0], -best[1]):
                best = (len(path) - 1, i)
    return best


def test_greedy_tree_matches_brute_force():
    from synthetic import tree_parents
    rng = np.random.default_rng(11)
    par = tree_parents([4, 2, 2])
    assert len(par) == 29
    assert list(par[1:5]) == [0] * 4
    assert list(par[5:13]) == [1 + (i - 5) // 2 for i in range(5, 13)]
    assert list(par[13:]) == [5 + (i - 13) // 2 for i in range(13, 29)]
    V = 3
    for trial in range(300):
        logits = rng.standard_normal((29, V))
        toks = rng.integers(0, V, 29)
        depth, node, path, nxt = A.accept_greedy_tree(toks, par, logits)
        bd, bn = _brute_tree(toks, par, logits)
        assert (depth, node) == (bd, bn)
        assert path[0] == 0 and path[-1] == node and len(path) == depth + 1
        assert nxt == int(np.argmax(logits[node]))


def test_tree_with_unit_branching_is_chain():
    from synthetic import tree_parents
    par = tree_parents([1, 1, 1, 1])
    assert list(par) == [-1, 0, 1, 2, 3]
    rng = np.random.default_rng(5)
    for _ in range(50):
        logits = rng.standard_normal((5, 4))
        toks = rng.integers(0, 4, 5)
        d, node, path, nxt = A.accept_greedy_tree(toks, par, logits)
        assert (d, nxt) == A.accept_greedy_chain(toks[1:], logits)
        assert path == list(range(d + 1))


def test_commit_tree_moves_in_place():
    from synthetic import tree_parents
    par = tree_parents([4, 2, 2])
    rng = np.random.default_rng(2)
    for node in range(29):
        path = A.tree_path(par, node)
        s = 10
        moves, n = A.commit_tree_moves(s, path)
        assert n == s + len(path)
        buf = rng.standard_normal((s + 29, 3))
        snap = buf.copy()
        for src, dst in moves:
            buf[dst] = buf[src]
        for d, row in enumerate(path):
            np.testing.assert_array_equal(buf[s + d], snap[s + row])
        np.testing.assert_array_equal(buf[:s], snap[:s])


def test_commit_chain_length():
    assert A.commit_chain(100, 0) == 101 and A.commit_chain(100, 4) == 105


def test_schedule_hand_table():
    assert A.next_k(0.3) == 2
    assert A.next_k(0.55) == 9
    assert A.next_k(0.8) == 16
    assert A.next_k(0.95) == 16
    assert A.next_k(0.0) == 2
    assert A.confidence(1.0, 1.0, 1.0) == pytest.approx(1.0)
    assert A.confidence(0.5, 0.05, 0.5) == pytest.approx(0.4 * 0.5 + 0.3 * 0.25 + 0.3 * 0.5)


def test_schedule_update_ema():
    k, ema, c = A.schedule_update(0.5, 4, 4, [0.9] * 5, [0.05] * 5)
    assert ema == pytest.approx(0.55)
    assert c == pytest.approx(0.4 * 0.9 + 0.3 * 1.0 + 0.3 * 0.55)
    assert k == 16
    k, ema, c = A.schedule_update(0.5, 0, 2, [0.01] * 3, [0.005] * 3)
    assert ema == pytest.approx(0.45) and k == 2


def test_mean_emitted_matches_overlap_product():
    """Monte Carlo: mean tokens per round = 1 + sum_j prod_{i<=j} beta_i (4 sigma)."""
    from synthetic import make_accept_inputs
    B, k, V = 600, 3, 64
    p, q, x, u = make_accept_inputs(B, k, V, seed=9, sigma=1.0, noise=0.7)
    emitted = np.array([A.accept_sampling_chain(p[b], q[b], x[b], u[b])[0] + 1 for b in range(B)])
    beta = np.minimum(p[:, :k].astype(np.float64), q.astype(np.float64)).sum(-1)   # [B, k]
    want = np.array([expected_tokens_positional(beta[b]) for b in range(B)])
    var = np.var(emitted)
    assert abs(emitted.mean() - want.mean()) < 4 * np.sqrt(var / B) + 1e-9


# -- temperature and top-p ----------------------------------------------------
def test_probs_at_two_tokens_is_logistic():
    """Two tokens: p0 = 1 / (1 + exp((l1 - l0) / T)) (closed form)."""
    for l0, l1, T in [(0.3, -1.2, 1.0), (2.0, 2.5, 0.7), (-4.0, 3.0, 2.5), (1.0, 1.0, 0.3)]:
        p = A.probs_at(np.array([l0, l1]), T)
        want = 1.0 / (1.0 + np.exp((l1 - l0) / T))
        assert abs(float(p[0]) - want) <= 2.0 ** -24 and abs(float(p[1]) - (1 - want)) <= 2.0 ** -24


def test_probs_at_ratios_follow_temperature():
    """p_x / p_y = exp((l_x - l_y) / T) up to float32 rounding of both."""
    rng = np.random.default_rng(3)
    lg = rng.standard_normal(50) * 2.0
    for T in (0.5, 1.0, 1.7):
        p = A.probs_at(lg, T).astype(np.float64)
        for x, y in [(0, 1), (7, 30), (12, 49)]:
            assert p[x] / p[y] == pytest.approx(np.exp((lg[x] - lg[y]) / T), rel=4e-7)
        assert abs(p.sum() - 1.0) < 50 * 2.0 ** -24


def test_probs_at_cold_temperature_is_one_hot():
    lg = np.array([0.1, 0.4, 0.39, -2.0])
    p = A.probs_at(lg, 1e-5)            # the nearest gap is 1000 temperatures
    assert list(p) == [0.0, 1.0, 0.0, 0.0]
    with pytest.raises(ValueError):
        A.probs_at(lg, 0.0)


def test_top_p_hand_example():
    """0.4 + 0.3 reaches 0.5 and 0.4 alone does not: nucleus {1, 3}, renormalised 4/7, 3/7."""
    p = np.array([0.1, 0.4, 0.2, 0.3], dtype=np.float32)
    assert list(A.top_p_keep(p, 0.5)) == [False, True, False, True]
    f = A.top_p_filter(p, 0.5)
    np.testing.assert_allclose(f, [0.0, 4 / 7, 0.0, 3 / 7], rtol=2e-7, atol=0)
    assert list(A.top_p_keep(p, 0.75)) == [False, True, True, True]
    assert A.top_p_keep(p, 1.0).all()
    np.testing.assert_array_equal(A.top_p_filter(p, 1.0), p / np.float32(p.astype(np.float64).sum()))


def test_top_p_ties_go_to_lower_ids():
    p = np.full(4, 0.25, dtype=np.float32)
    assert list(A.top_p_keep(p, 0.5)) == [True, True, False, False]
    assert list(A.top_p_keep(p, 0.5 + 2.0 ** -24)) == [True, True, True, False]
    assert list(A.top_p_keep(p, 2.0 ** -24)) == [True, False, False, False]


def test_top_p_smallest_keeps_the_argmax():
    rng = np.random.default_rng(5)
    p = _rand_rows(rng, 40, 1)[0]
    keep = A.top_p_keep(p, 2.0 ** -24)
    assert keep.sum() == 1 and keep[int(np.argmax(p))]


@pytest.mark.parametrize("seed", range(4))
def test_top_p_nucleus_properties(seed):
    """The nucleus is characterised without the oracle's sort: it is closed upward
    (any token ranked above a kept one is kept), its exact mass fraction reaches
    top_p, and dropping its lowest-ranked token falls below top_p."""
    rng = np.random.default_rng(seed)
    V = 8
    for row in _rand_rows(rng, V, 20):
        if seed == 3:
            row[:3] = row[3]                                  # ties
        w = [int(x) for x in A.int_weights(row)]
        S = sum(w)
        for m in rng.integers(1, TWO24, size=6):
            top_p = float(np.float32(int(m) * 2.0 ** -24))
            keep = A.top_p_keep(row, top_p)
            K = [x for x in range(V) if keep[x]]
            above = lambda y, x: row[y] > row[x] or (row[y] == row[x] and y < x)
            for x in K:
                assert all(keep[y] for y in range(V) if above(y, x))
            goal = Fraction(int(m), TWO24)
            assert Fraction(sum(w[x] for x in K), S) >= goal
            last = max(K, key=lambda x: (-float(row[x]), x))
            assert Fraction(sum(w[x] for x in K) - w[last], S) < goal


@pytest.mark.parametrize("seed", [0, 1])
def test_top_p_rejection_law_equals_nucleus(seed):
    """Target truncated to its nucleus, draft left whole: the emitted token's law
    is the renormalised nucleus (k = 1, V = 5, exact over all uniforms)."""
    rng = np.random.default_rng(10 + seed)
    V = 5
    p_full = _rand_rows(rng, V, 2)
    p = np.stack([A.top_p_filter(r, 0.7) for r in p_full])
    assert (p[0] == 0).any()
    q = _rand_rows(rng, V, 1)
    first = [0.0] * V
    for x in range(V):
        qx = float(q[0, x])
        keep_end = _first_true(lambda m: not A.ratio_accept(_u(m), q[0, x], p[0, x]))
        first[x] += qx * keep_end / TWO24
        if keep_end < TWO24:
            law = _sampler_law_of(lambda m: A.accept_sampling_chain(p, q, [x], [_u(keep_end), _u(m)])[1], V)
            for y in range(V):
                first[y] += qx * (1 - keep_end / TWO24) * law[y]
    tol = 4 * 2.0 ** -24 + V * 2.0 ** -30 + V * 2.0 ** -23
    np.testing.assert_allclose(first, p[0].astype(np.float64), rtol=0, atol=tol)
    assert all(first[y] == 0.0 for y in range(V) if p[0, y] == 0)


# -- alternative draft-length schedules ----------------------------------------
def test_first_reject_resets_to_min():
    """DSpark refinement: a round whose first draft token is rejected drops k to
    min_k whatever the confidence; otherwise the linear map decides."""
    sch = A.KSchedule(first_reject_min=True)
    top1, top2 = [0.99] * 5, [0.001] * 5          # confidence high enough for max_k
    k0, _, c0 = A.schedule_update(0.9, 0, 4, top1, top2, A.KSchedule())
    k1, _, c1 = A.schedule_update(0.9, 0, 4, top1, top2, sch)
    assert c0 == c1 and k0 > sch.min_k and k1 == sch.min_k
    k2, _, _ = A.schedule_update(0.9, 1, 4, top1, top2, sch)
    assert k2 == A.schedule_update(0.9, 1, 4, top1, top2, A.KSchedule())[0] > sch.min_k


def test_aimd_hand_sequence():
    """All kept: +1 a round up to 8; all rejected: the window's acceptance falls
    below 0.7 after enough rounds, then -1 a round down to 2."""
    h, k, ks = [], 2, []
    for _ in range(8):
        k, h = A.aimd_update(h, k, k)
        ks.append(k)
    assert ks == [3, 4, 5, 6, 7, 8, 8, 8]
    # 8 rounds of 8/8 then rejections of k: window acceptance = kept / drafted
    ks = []
    for _ in range(6):
        k, h = A.aimd_update(h, 0, k)
        ks.append(k)
    kept = sum(a for a, _ in h)
    assert kept == 2 + 3 + 4 + 5 + 6 + 7 + 8 + 8
    # acceptance after each rejection round: 43/(43+8), 43/(43+16), 43/(43+23), ...
    # 43/51 = 0.843 (keep), 43/59 = 0.729 (keep), 43/66 = 0.652 (-1) ...
    assert ks[:3] == [8, 8, 7]
    assert ks[-1] < 7


def test_aimd_thresholds_are_strict_and_window_slides():
    sch = A.AIMDSchedule(window=4)
    # 17 of 20 kept is exactly 0.85: no change; 7 of 10 exactly 0.7: no change
    k, h = A.aimd_update([(5, 5), (5, 5), (5, 5)], 2, 5, sch)
    assert k == 5 and len(h) == 4
    k, h = A.aimd_update([(5, 10), (2, 0)], 0, 0, A.AIMDSchedule(window=4, min_k=0))
    assert k == 0          # 7/10 exactly: unchanged
    # the window forgets: after 4 perfect rounds the early failures are gone
    h = [(0, 8)] * 4
    for _ in range(4):
        k, h = A.aimd_update(h, 8, 8, A.AIMDSchedule(window=4))
    assert h == [(8, 8)] * 4 and k == 8


def test_decay_k_table():
    """K_t = max(1, round(6 (1 - t/100))): halves round to even."""
    want = {0: 6, 10: 5, 25: 4, 50: 3, 75: 2, 90: 1, 99: 1, 100: 1, 150: 1}
    for t, k in want.items():
        assert A.decay_k(t, 100, 6) == k, (t, A.decay_k(t, 100, 6))
    assert A.decay_k(1, 8, 4) == 4          # 3.5 -> 4 (even)
    assert A.decay_k(3, 8, 4) == 2          # 2.5 -> 2 (even)


# -- top-1 / top-2 probabilities of the confidence score (DSpark page, 0539edu.com/news/4524681, §2.2) --
def test_top12_two_logits_is_logistic():
    # two tokens: p(top) = 1 / (1 + e^-(l0 - l1)), p(second) = 1 - p(top)
    for l0, l1 in [(1.5, -0.25), (0.0, 3.0), (-7.0, -7.5)]:
        p1, p2 = A.top12_probs([l0, l1])
        hi, lo = max(l0, l1), min(l0, l1)
        want = 1.0 / (1.0 + np.exp(-(hi - lo)))
        assert abs(p1 - want) < 1e-15 and abs(p2 - (1.0 - want)) < 1e-15


def test_top12_hand_row_with_log_integer_logits():
    # logits log(4), log(2), log(1), log(1): probabilities 4/8, 2/8, 1/8, 1/8 whatever the order
    row = np.log(np.array([1.0, 4.0, 1.0, 2.0]))
    p1, p2 = A.top12_probs(row)
    assert abs(p1 - 0.5) < 1e-15 and abs(p2 - 0.25) < 1e-15
    # a constant shift of every logit changes nothing
    q1, q2 = A.top12_probs(row + 40.0)
    assert abs(q1 - 0.5) < 1e-14 and abs(q2 - 0.25) < 1e-14


def test_top12_tie_at_the_top_counts_both():
    # the two largest logits tie: both probabilities are e^0 / sum = 2 / (2 + e^-1 + e^-2)
    row = [0.0, 3.0, 2.0, 3.0, 1.0]
    p1, p2 = A.top12_probs(row)
    want = 1.0 / (2.0 + np.exp(-1.0) + np.exp(-2.0) + np.exp(-3.0))
    assert abs(p1 - want) < 1e-15 and p1 == p2


def test_top12_uniform_row():
    for V in (2, 7, 1024):
        p1, p2 = A.top12_probs(np.full(V, -1.25))
        assert abs(p1 - 1.0 / V) < 1e-15 and abs(p2 - 1.0 / V) < 1e-15


def test_top12_are_probabilities_not_logits():
    # a clear winner: top1 near 1, top2 the second probability, both in (0, 1]
    row = [10.0, 0.0, -1.0]
    p1, p2 = A.top12_probs(row)
    S = 1.0 + np.exp(-10.0) + np.exp(-11.0)
    assert abs(p1 - 1.0 / S) < 1e-15 and abs(p2 - np.exp(-10.0) / S) < 1e-18
    assert 0.0 < p2 < p1 <= 1.0
