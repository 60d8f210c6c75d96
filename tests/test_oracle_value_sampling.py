"""Pins of the oracle's value-row sampling (CPU).

Value rows are drawn inside each selected team from the group-mean in-team softmax r_j, and
head g weighs row j by exp(s_gj - m) / r_j ("Stochastic Sparse Attention for Memory-Bound
Inference", abstract: sample value rows from the post-softmax distribution and gather-add
them).  Pins: r against numpy softmax of independently decoded keys; the expectation over
every sequence of row draws against the full P.V sums; draw frequencies; Monte Carlo over
seeds; and convergence to the full-team estimate with many rows.
"""
import itertools

import numpy as np
import pytest

import oracle
from sampled_sparse_decode_gb300 import workloads as W
from test_oracle import _decoded, _problem, _tiny


def _team_tokens(wl, b, h, team):
    T = wl.cfg.team_size
    L = int(wl.seq_lens[b])
    page = wl.page_table[b, team]
    n = min(T, L - team * T)
    return _decoded(wl.k_pool[page, h, :n]), _decoded(wl.v_pool[page, h, :n])


@pytest.mark.parametrize("G", [1, 2, 3])
def test_row_probs_are_the_group_mean_team_softmax(G):
    wl = W.generate(_tiny(seq_len=30, team_size=8, head_dim=8, q_heads=2 * G, kv_heads=2,
                          data_seed=4), invalid_fill=float("nan"))
    pr = _problem(wl)
    for h in range(2):
        for team in range(4):
            K, _ = _team_tokens(wl, 0, h, team)
            q = _decoded(wl.q[0, h * G:(h + 1) * G])
            s = q @ K.T / np.sqrt(8)
            sm = np.exp(s - s.max(axis=1, keepdims=True))
            sm /= sm.sum(axis=1, keepdims=True)
            np.testing.assert_allclose(oracle.vs_row_probs(pr, 0, h, team), sm.mean(axis=0),
                                       rtol=1e-13)


@pytest.mark.parametrize("S", [1, 2, 3])
def test_expectation_over_row_draws_equals_full_team_sums(S):
    """For each team, the expectation over all len^S row-draw sequences (probability
    prod r) of the sampled numerator equals the full P.V numerator; the denominator is
    exact.  Partial last team, G = 2, Horvitz-Thompson weights."""
    wl = W.generate(_tiny(seq_len=11, team_size=4, head_dim=4, q_heads=2, kv_heads=1,
                          data_seed=9), invalid_fill=float("nan"))
    pr = _problem(wl)
    sel = np.array([0, 2], np.int32)                   # team 2 is partial (3 tokens)
    pi = np.array([0.4, 0.9])
    shift = np.array([0.2, -0.1])
    full_num, full_den = oracle.num_den(pr, 0, 0, sel, pi, shift)
    E_num = np.zeros_like(full_num)
    for c, team in enumerate(sel):
        r = oracle.vs_row_probs(pr, 0, 0, int(team))
        for seq in itertools.product(range(r.size), repeat=S):
            num, den = oracle.num_den_vs(pr, 0, 0, sel[c:c + 1], pi[c:c + 1], S,
                                         np.array(seq, np.int32), shift)
            E_num += np.prod(r[list(seq)]) * num
            np.testing.assert_allclose(den, oracle.num_den(pr, 0, 0, sel[c:c + 1],
                                                           pi[c:c + 1], shift)[1], rtol=1e-14)
    np.testing.assert_allclose(E_num, full_num, rtol=1e-12, atol=1e-13)


def test_row_draw_frequencies_follow_r():
    wl = W.generate(_tiny(seq_len=64, team_size=16, head_dim=8, q_heads=2, kv_heads=1,
                          data_seed=2))
    pr = _problem(wl)
    r = oracle.vs_row_probs(pr, 0, 0, 1)
    counts = np.zeros(r.size)
    for seed in range(400):
        idx, t, C = oracle.vs_draw(pr, 0, 0, 1, 64, seed)
        counts += np.bincount(idx, minlength=r.size)
    N = counts.sum()
    chi2 = ((counts - N * r) ** 2 / (N * r)).sum()
    assert chi2 < r.size - 1 + 6 * np.sqrt(2 * (r.size - 1))     # ~6 sigma


def test_monte_carlo_unbiased_numerator():
    """Over 2048 seeds, the mean of <num_vs, w> lies within 3.5 standard errors of the full
    numerator, with the team draws fixed."""
    wl = W.generate("tiny_f32")
    pr = _problem(wl)
    sel = np.array([1, 5, 9, 20], np.int32)
    pi = np.array([0.3, 0.5, 0.7, 1.0])
    shift = np.array([1.0, 1.5])
    full_num, _ = oracle.num_den(pr, 0, 0, sel, pi, shift)
    w = np.random.default_rng(3).standard_normal(64)
    est = []
    for seed in range(2048):
        idx = np.concatenate([oracle.vs_draw(pr, 0, 0, int(t), 4, seed)[0] for t in sel])
        num, _ = oracle.num_den_vs(pr, 0, 0, sel, pi, 4, idx, shift)
        est.append(num @ w)
    est = np.array(est)
    se = est.std(axis=0, ddof=1) / np.sqrt(est.shape[0])
    assert (np.abs(est.mean(axis=0) - full_num @ w) < 3.5 * se).all()


def test_many_rows_approach_the_full_team_estimate():
    wl = W.generate("tiny_f32")
    pr = _problem(wl)
    sel = np.array([0, 3, 7], np.int32)
    pi = np.array([0.5, 0.6, 0.8])
    full = oracle.attend(pr, 0, 0, sel, pi)
    out, idx = oracle.attend_vs(pr, 0, 0, sel, pi, 4096, 11)
    assert idx.shape == (3, 4096) and (idx >= 0).all() and (idx < 64).all()
    assert np.abs(out - full).max() < 0.05 * np.abs(full).max() + 0.02


def test_row_draw_uses_counter_k_h_b_one_plus_team():
    """Row draw k of team i of unit (b, h) uses Philox word 0 of counter (k, h, b, 1 + i)
    (the Philox function itself is pinned against an independent implementation)."""
    Z = (1 << 62) + 12345
    for seed, b, h, team, k in [(0, 0, 0, 0, 0), (7, 3, 1, 5, 9), (2 ** 40 + 3, 1, 2, 200, 63)]:
        x = int(oracle.philox4x32_10([k, h, b, 1 + team], [seed & 0xFFFFFFFF, seed >> 32])[0])
        assert oracle.lib().oracle_vs_point(seed, b, h, team, k, Z) == ((2 * x + 1) * Z) >> 33
