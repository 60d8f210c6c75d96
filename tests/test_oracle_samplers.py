"""Pins of the oracle's sampler variants (CPU): systematic draws with Horvitz-Thompson
weights, i.i.d. draws with Hansen-Hurwitz weights, and the defensive uniform mixture.

Systematic: one uniform u, points (r + u) / M on the CDF; team i is hit with probability
min(1, M q_i) (stratified / systematic variants, "Stochastic Sparse Attention for
Memory-Bound Inference", abstract).  Hansen-Hurwitz: weight c_i / (M q_i) per drawn team
(the per-draw 1/p_i reweighting of the explainer, section 三 step 5).  Mixture:
q = (1 - alpha) p + alpha / n (explainer, section 八, pitfall 4).  Each function is checked
against exact fractions, brute force over the uniform, enumeration of draw sequences or the
dense special case: never against a retyped copy of its own formula.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from sampled_sparse_decode_gb300 import workloads as W
from test_oracle import _dense_numpy, _decoded, _problem, _tiny, _unit_tokens


def _unit_p(seq_len=19, team_size=4, data_seed=3):
    cfg = _tiny(seq_len=seq_len, team_size=team_size, head_dim=4, q_heads=2, kv_heads=1,
                data_seed=data_seed)
    wl = W.generate(cfg, invalid_fill=float("nan"))
    pr = _problem(wl)
    reps = oracle.build_reps(pr, wl.page_fill)
    return wl, pr, reps, oracle.team_probs(pr, reps, 0, 0)


def test_mixture_is_a_distribution_with_a_uniform_floor():
    _, _, _, p = _unit_p()
    n = p.size
    for alpha in (0.0, 0.05, 0.3, 1.0):
        q = oracle.mix(p, alpha)
        assert abs(q.sum() - 1.0) < 1e-14
        assert (q >= alpha / n * (1 - 1e-14)).all()
    np.testing.assert_array_equal(oracle.mix(p, 0.0), p)
    np.testing.assert_allclose(oracle.mix(p, 1.0), np.full(n, 1.0 / n), rtol=1e-15)
    # a team the scores nearly exclude keeps at least alpha / n
    spiky = np.array([1.0 - 3e-12, 1e-12, 1e-12, 1e-12])
    assert oracle.mix(spiky, 0.05)[1] >= 0.05 / 4


def test_systematic_points_are_floor_of_exact_fractions():
    """floor((r Z + floor(u Z)) / M) equals floor((r + u) Z / M) with u = (2x + 1) / 2^33
    evaluated in exact rational arithmetic."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        Z = int(rng.integers(1, 2 ** 62)) + (1 << 62) * int(rng.integers(0, 2))
        Z = min(Z, (1 << 63) - 1)
        M = int(rng.integers(1, 4097))
        x = int(rng.integers(0, 2 ** 32))
        u = Fraction(2 * x + 1, 2 ** 33)
        t_u = (u * Z).numerator // (u * Z).denominator
        for r in (0, M // 2, M - 1):
            want = Fraction(r) + u
            want = (want * Z / M)
            assert oracle.systematic_point(t_u, r, M, Z) == want.numerator // want.denominator
            assert oracle.systematic_point(t_u, r, M, Z) < Z


def _grid_selection(q, M, K=4096):
    """For u on the midpoints of a K-grid: the teams hit by the systematic points, via the
    oracle's point and CDF-search routines.  Returns the hit-count matrix [K][n]."""
    n = q.size
    C = np.cumsum([oracle.fixed_prob(v) for v in q]).astype(np.uint64)
    Z = int(C[-1])
    hits = np.zeros((K, n), dtype=np.int64)
    for k in range(K):
        t_u = ((2 * k + 1) * Z) // (2 * K)             # floor(u Z), u = (k + 1/2) / K
        for r in range(M):
            i = oracle.cdf_search(C, oracle.systematic_point(t_u, r, M, Z))
            hits[k, i] += 1
    return hits


def test_systematic_inclusion_is_min_one_Mq_by_brute_force():
    _, _, _, p = _unit_p()
    q = oracle.mix(p, 0.1)
    for M in (1, 2, 3, 7):
        hits = _grid_selection(q, M)
        freq = (hits > 0).mean(axis=0)
        np.testing.assert_allclose(freq, np.minimum(1.0, M * q), atol=2.0 / 4096)
        # every team is hit floor(M q_i) or ceil(M q_i) times, and M times in total
        assert (hits.sum(axis=1) == M).all()
        lo, hi = np.floor(M * q - 1e-9), np.ceil(M * q + 1e-9)
        assert ((hits >= lo) & (hits <= hi)).all()
        # the oracle's weights are these inclusion probabilities
        for k in (0, 1000, 4095):
            draws = np.repeat(np.arange(q.size, dtype=np.int32), hits[k])
            sel, rc = oracle.select_ex(draws, q, "systematic")
            assert np.array_equal(sel, np.nonzero(hits[k])[0])
            np.testing.assert_allclose(rc, freq[sel], atol=2.0 / 4096)


def test_systematic_horvitz_thompson_is_unbiased_over_u():
    _, _, _, p = _unit_p()
    q = oracle.mix(p, 0.05)
    f = np.random.default_rng(1).uniform(0.5, 2.0, size=q.size)
    for M in (2, 3):
        K = 4096
        hits = _grid_selection(q, M, K)
        est = []
        for k in range(K):
            draws = np.repeat(np.arange(q.size, dtype=np.int32), hits[k])
            sel, rc = oracle.select_ex(draws, q, "systematic")
            est.append((f[sel] / rc).sum())
        assert abs(np.mean(est) - f.sum()) < 4.0 / K * f.sum() * M


@pytest.mark.parametrize("M,alpha", [(1, 0.0), (2, 0.0), (3, 0.0), (3, 0.2)])
def test_hansen_hurwitz_expectation_by_enumeration(M, alpha):
    """Over all n^M ordered draw sequences, E[sum_S c_i f_i / (M q_i)] = sum f_i exactly;
    and with the oracle's attention sums: E[num], E[den] equal the dense sums."""
    wl, pr, reps, p = _unit_p()
    q = oracle.mix(p, alpha)
    n = q.size
    f = np.random.default_rng(2).uniform(0.5, 2.0, size=n)
    shift = np.array([0.1, -0.4])
    E_f, E_num, E_den = 0.0, np.zeros((2, 4)), np.zeros(2)
    for seq in itertools.product(range(n), repeat=M):
        prob = np.prod(q[list(seq)])
        sel, rc = oracle.select_ex(np.array(seq, np.int32), q, "iid_hh")
        E_f += prob * (f[sel] / rc).sum()
        num, den = oracle.num_den(pr, 0, 0, sel, rc, shift)
        E_num += prob * num
        E_den += prob * den
    assert abs(E_f - f.sum()) < 1e-12 * f.sum()
    K, V = _unit_tokens(wl, 0, 0)
    e = np.exp(_decoded(wl.q[0]) @ K.T / 2.0 - shift[:, None])
    np.testing.assert_allclose(E_den, e.sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(E_num, e @ V, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("M,alpha", [(2, 0.0), (3, 0.25)])
def test_mixed_horvitz_thompson_expectation_by_enumeration(M, alpha):
    """The i.i.d. Horvitz-Thompson weights stay unbiased when the draws follow the mixture."""
    wl, pr, reps, p = _unit_p()
    q = oracle.mix(p, alpha)
    shift = np.array([0.0, 0.2])
    E_num, E_den = np.zeros((2, 4)), np.zeros(2)
    for seq in itertools.product(range(q.size), repeat=M):
        prob = np.prod(q[list(seq)])
        sel, rc = oracle.select_ex(np.array(seq, np.int32), q, "iid_ht")
        num, den = oracle.num_den(pr, 0, 0, sel, rc, shift)
        E_num += prob * num
        E_den += prob * den
    K, V = _unit_tokens(wl, 0, 0)
    e = np.exp(_decoded(wl.q[0]) @ K.T / 2.0 - shift[:, None])
    np.testing.assert_allclose(E_den, e.sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(E_num, e @ V, rtol=1e-12, atol=1e-12)


def test_decode_ex_defaults_are_the_plain_method():
    wl = W.generate(_tiny(seq_len=100, team_size=8, head_dim=16, q_heads=4, kv_heads=2,
                          dtype="bf16"))
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    for h in range(2):
        a = oracle.decode(pr, reps, 6, 42, 0, h)
        b = oracle.decode_ex(pr, reps, 6, 42, 0, h, "iid_ht", 0.0)
        assert np.array_equal(a.draws, b.draws) and np.array_equal(a.sel, b.sel)
        np.testing.assert_array_equal(a.pi, b.pi)
        np.testing.assert_array_equal(a.p, b.p)
        np.testing.assert_array_equal(a.out, b.out)


def test_uniform_systematic_with_M_equal_n_is_dense_attention():
    """alpha = 1 makes q uniform; with M = n systematic points every team is hit exactly
    once with pi = 1, so the estimate is dense softmax attention."""
    wl = W.generate("tiny_f32")
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    n = wl.cfg.n_teams
    r = oracle.decode_ex(pr, reps, n, 3, 0, 0, "systematic", 1.0)
    assert r.sel.size == n and (r.pi == 1.0).all()
    assert sorted(r.draws.tolist()) == list(range(n))
    np.testing.assert_allclose(r.out, _dense_numpy(wl, 0, 0), rtol=0, atol=1e-12)


def test_systematic_draws_follow_Mq():
    wl = W.generate("tiny_f32")
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    p = oracle.team_probs(pr, reps, 0, 0)
    for seed in range(20):
        for alpha in (0.0, 0.1):
            q = oracle.mix(p, alpha)
            draws, t, C = oracle.draw_systematic(q, 8, seed, 0, 0)
            assert (np.diff(draws) >= 0).all()                      # points are ordered
            c = np.bincount(draws, minlength=q.size)
            assert ((c >= np.floor(8 * q - 1e-9)) & (c <= np.ceil(8 * q + 1e-9))).all()
            # the first point is the i.i.d. sampler's draw 0 scaled by 1/M
            assert t[0] == int(oracle.draw(q, 1, seed, 0, 0)[1][0]) // 8


@pytest.mark.parametrize("sampler,alpha", [("systematic", 0.0), ("iid_hh", 0.0),
                                           ("iid_ht", 0.1)])
def test_monte_carlo_unbiased_num_and_den_per_sampler(sampler, alpha):
    """Over 2048 seeds of the tiny fp32 workload (M = 8), the means of the weighted
    denominator and of <numerator, w> lie within 3.5 standard errors of the dense values."""
    wl = W.generate("tiny_f32")
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    q = oracle.mix(oracle.team_probs(pr, reps, 0, 0), alpha)
    K, V = _unit_tokens(wl, 0, 0)
    s = _decoded(wl.q[0]) @ K.T / 8.0
    shift = s.max(axis=1)
    e = np.exp(s - shift[:, None])
    w = np.random.default_rng(0).standard_normal(64)
    w /= np.linalg.norm(w)
    dens, nums = [], []
    for seed in range(2048):
        draws, _, _ = oracle.draw_with(sampler, q, 8, seed, 0, 0)
        sel, rc = oracle.select_ex(draws, q, sampler)
        num, den = oracle.num_den(pr, 0, 0, sel, rc, shift)
        dens.append(den)
        nums.append(num @ w)
    for est, truth in [(np.array(dens), e.sum(axis=1)), (np.array(nums), (e @ V) @ w)]:
        se = est.std(axis=0, ddof=1) / np.sqrt(est.shape[0])
        assert (np.abs(est.mean(axis=0) - truth) < 3.5 * se).all()
