"""Holding a sampled team set over several decode steps (the explainer's pitfall 2 on
variance accumulating over autoregressive steps: fix the team assignment for a stretch of
steps, e.g. refresh every 256).

The reading pinned here: the set S and its inclusion probabilities pi are drawn once, from
the query and cache of the refresh step.  Later steps reuse them with their own query on
the grown cache.  Horvitz-Thompson stays unbiased for any per-team quantity, so a later
step's numerator and denominator are still unbiased for the dense sums over every team that
existed at the refresh step.  That includes tokens appended to those teams later.  A team
opened after the refresh has pi = 0 and is missing until the next refresh.  Both facts are
checked by enumerating every ordered draw sequence on tiny inputs, against plain numpy sums,
and by a hand-derived example in exact rationals (tests/golden/worked_held_set.txt).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from sampled_sparse_decode_gb300 import workloads as W


def _cfg(**kw):
    base = dict(batch=1, q_heads=2, kv_heads=1, head_dim=4, seq_len=24, team_size=4, draws=3,
                keys="gauss", heavy_rate=0.0, paged=False, num_pages=0, data_seed=5,
                dtype="f32")
    base.update(kw)
    return W.Config("held", **base)


def _tokens(wl, L):
    """The first L keys and values of unit (0, 0) in token order, float64."""
    T = wl.cfg.team_size
    K = np.concatenate([wl.k_pool[wl.page_table[0, i], 0] for i in range(-(-L // T))])
    V = np.concatenate([wl.v_pool[wl.page_table[0, i], 0] for i in range(-(-L // T))])
    return K[:L].astype(np.float64), V[:L].astype(np.float64)


def _expectations(wl, L0, L1, q_later, M, shift):
    """Exact E[num] and E[den] at a later step (query q_later, length L1) over every ordered
    draw sequence of the refresh step (the workload's own query, length L0)."""
    T = wl.cfg.team_size
    fill0 = np.zeros(wl.k_pool.shape[0], np.int32)
    for i in range(-(-L0 // T)):
        fill0[wl.page_table[0, i]] = min(T, L0 - i * T)
    pr0 = oracle.Problem(wl.q, wl.k_pool, wl.v_pool, wl.page_table, np.array([L0], np.int32))
    p = oracle.team_probs(pr0, oracle.build_reps(pr0, fill0), 0, 0)
    pr1 = oracle.Problem(q_later, wl.k_pool, wl.v_pool, wl.page_table,
                         np.array([L1], np.int32))
    G, d = wl.cfg.group, wl.cfg.head_dim
    E_num, E_den = np.zeros((G, d)), np.zeros(G)
    for seq in itertools.product(range(p.size), repeat=M):
        prob = np.prod(p[list(seq)])
        sel, pi = oracle.select(np.array(seq, np.int32), p)
        num, den = oracle.num_den(pr1, 0, 0, sel, pi, shift)
        E_num += prob * num
        E_den += prob * den
    return p.size, E_num, E_den


@pytest.mark.parametrize("M", [1, 3])
def test_held_set_stays_unbiased_for_a_later_query_on_grown_teams(M):
    """Five teams at the refresh step (the last one partial, 2 of 4 tokens); the later step
    has a different query and two more tokens in that last team."""
    L0, L1 = 18, 20
    wl = W.generate(_cfg(), seq_lens=[24], invalid_fill=float("nan"))
    q_later = np.random.default_rng(8).standard_normal(wl.q.shape).astype(np.float32)
    shift = np.array([0.4, -0.1])
    n0, E_num, E_den = _expectations(wl, L0, L1, q_later, M, shift)
    assert n0 == 5
    K, V = _tokens(wl, L1)
    e = np.exp(q_later[0].astype(np.float64) @ K.T / np.sqrt(4.0) - shift[:, None])
    np.testing.assert_allclose(E_den, e.sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(E_num, e @ V, rtol=1e-12, atol=1e-12)


def test_team_opened_after_the_refresh_is_missing_until_the_next():
    """The later step's cache has a sixth team (one token): the held design never selects
    it, so the expectations equal the dense sums over the first five teams only, and
    differ from the sums over all tokens by exactly that token's terms."""
    L0, L1 = 20, 21
    wl = W.generate(_cfg(), seq_lens=[24], invalid_fill=float("nan"))
    q_later = np.random.default_rng(9).standard_normal(wl.q.shape).astype(np.float32)
    shift = np.zeros(2)
    n0, E_num, E_den = _expectations(wl, L0, L1, q_later, 2, shift)
    assert n0 == 5
    K, V = _tokens(wl, L1)
    e = np.exp(q_later[0].astype(np.float64) @ K.T / 2.0)
    np.testing.assert_allclose(E_den, e[:, :20].sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(E_num, e[:, :20] @ V[:20], rtol=1e-12, atol=1e-12)
    assert np.all(np.abs(E_den - e.sum(axis=1)) >= 0.5 * e[:, 20])


def _golden(name):
    vals = {}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    for line in open(path):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = np.array([float(x) for x in v.split()])
    return vals


def test_worked_held_set_example():
    """Hand-derived example (tests/golden/worked_held_set.txt): the two-team problem sampled
    with q = 1, then held for a later query q' = 2.  Per-outcome estimates and their exact
    expectations (the later query's dense sums)."""
    g = _golden("worked_held_set.txt")
    k = np.array(g["k"], np.float32).reshape(2, 1, 1, 1)
    v = np.array(g["v"], np.float32).reshape(2, 1, 1, 1)
    pt, lens = np.array([[0, 1]], np.int32), np.array([2], np.int32)
    pr0 = oracle.Problem(np.array([[[g["q"][0]]]], np.float32), k, v, pt, lens)
    p = oracle.team_probs(pr0, oracle.build_reps(pr0), 0, 0)
    M = int(g["M"][0])
    pi = np.array([oracle.select(np.full(M, i, np.int32), p)[1][0] for i in range(2)])
    np.testing.assert_allclose(pi, g["pi"], rtol=1e-6)
    pr1 = oracle.Problem(np.array([[[g["q_later"][0]]]], np.float32), k, v, pt, lens)
    got = {}
    for S, tag in [((0,), "S0"), ((1,), "S1"), ((0, 1), "S01")]:
        num, den = oracle.num_den(pr1, 0, 0, np.array(S, np.int32), pi[list(S)], 0.0)
        np.testing.assert_allclose([num[0, 0], den[0]], [g["num_" + tag][0], g["den_" + tag][0]],
                                   rtol=1e-6)
        got[S] = (num[0, 0], den[0])
    E_num = E_den = 0.0
    for seq in itertools.product(range(2), repeat=M):
        prob = np.prod(p[list(seq)])
        n_, d_ = got[tuple(sorted(set(seq)))]
        E_num += prob * n_
        E_den += prob * d_
    np.testing.assert_allclose([E_num, E_den], [g["E_num"][0], g["E_den"][0]], rtol=1e-6)
