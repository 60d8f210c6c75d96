"""Pins of the fp64 CPU oracle against facts fixed outside its own code.

Each test checks one step of SANTA++ ("SANTA++: Sampling Attention through Representative
Keys", abstract; explainer section 三 steps 1-5 and 3.1) against an independent source: a
library routine (Triton's Philox, torch's bf16 decoding and scaled_dot_product_attention),
a closed form or hand-derived value under tests/golden/, exact enumeration of all draw
sequences, or brute-force dense attention.
"""
import dataclasses
import itertools
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from sampled_sparse_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(wl: W.Workload) -> oracle.Problem:
    return oracle.Problem(wl.q, wl.k_pool, wl.v_pool, wl.page_table, wl.seq_lens)


def _decoded(a: np.ndarray) -> np.ndarray:
    """Stored elements as float64, decoded by torch (not by the oracle)."""
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
        return t.to(torch.float64).numpy()
    return a.astype(np.float64)


def _unit_tokens(wl: W.Workload, b: int, h: int):
    """All valid keys / values of unit (b, h) in token order, float64, via the page table."""
    T = wl.cfg.team_size
    L = int(wl.seq_lens[b])
    K = np.concatenate([_decoded(wl.k_pool[wl.page_table[b, i], h]) for i in range(-(-L // T))])
    V = np.concatenate([_decoded(wl.v_pool[wl.page_table[b, i], h]) for i in range(-(-L // T))])
    return K[:L], V[:L]


def _dense_numpy(wl, b, h):
    """Textbook softmax attention of the group's query heads over all valid tokens."""
    G, d = wl.cfg.group, wl.cfg.head_dim
    K, V = _unit_tokens(wl, b, h)
    q = _decoded(wl.q[b, h * G:(h + 1) * G])
    s = q @ K.T / np.sqrt(d)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w @ V) / w.sum(axis=1, keepdims=True)


def _tiny(**kw):
    base = dict(batch=1, q_heads=2, kv_heads=1, head_dim=8, seq_len=40, team_size=8, draws=4,
                keys="gauss", heavy_rate=0.0, paged=False, num_pages=0, data_seed=11, dtype="f32")
    base.update(kw)
    return W.Config("t", **base)


# ------------------------------------------------------------------ Philox and uniforms

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl
@triton.jit
def k(out, seed, c0p, c1p, c2p, c3p, N: tl.constexpr):
    o = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c0p + o), tl.load(c1p + o), tl.load(c2p + o), tl.load(c3p + o))
    tl.store(out + o * 4, a); tl.store(out + o * 4 + 1, b)
    tl.store(out + o * 4 + 2, c); tl.store(out + o * 4 + 3, d)
cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    c = torch.tensor(ctrs, dtype=torch.int64).to(torch.uint32)
    out = torch.zeros(4 * len(ctrs), dtype=torch.uint32)
    k[(1,)](out, seed, c[:, 0].contiguous(), c[:, 1].contiguous(), c[:, 2].contiguous(),
            c[:, 3].contiguous(), N=len(ctrs))
    res.append(out.to(torch.int64).tolist())
print(json.dumps(res))
"""


def test_philox_matches_triton_library():
    """Our Philox4x32-10 equals Triton's (an independent library implementation, run by its
    CPU interpreter) bit for bit, for 64-bit keys and counters with all four words set."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(5)
    seeds = [0, 1, 12345, 2**32 - 1, 2**32, 0x123456789ABCDEF, 2**63 - 1]
    cases = []
    for s in seeds:
        ctrs = rng.integers(0, 2**32, size=(16, 4), dtype=np.uint64)
        ctrs[0] = 0
        ctrs[1] = [7, 3, 1, 0]
        cases.append((int(s), ctrs.astype(np.int64).tolist()))
    r = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(cases),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    ref = json.loads(r.stdout.strip().splitlines()[-1])
    for (seed, ctrs), words in zip(cases, ref):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for j, c in enumerate(ctrs):
            got = oracle.philox4x32_10(c, key)
            assert list(map(int, got)) == words[4 * j:4 * j + 4], (seed, c)


def test_uniform_is_word0_of_counter_r_h_b():
    """u = (x0 + 1/2) / 2^32 with counter (r, h, b, 0) and key (lo32, hi32) of the seed."""
    for seed, b, h, r in [(0, 0, 0, 0), (99, 3, 2, 17), (2**40 + 5, 15, 7, 4095)]:
        x0 = int(oracle.philox4x32_10([r, h, b, 0], [seed & 0xFFFFFFFF, seed >> 32])[0])
        u = oracle.uniform(seed, b, h, r)
        assert u * 2.0**32 - 0.5 == x0
        assert 0.0 < u < 1.0


def test_uniforms_are_uniform():
    """Kolmogorov-Smirnov test of 20000 uniforms of one stream (fixed seed, deterministic)."""
    from scipy import stats
    u = np.array([oracle.uniform(1234, 2, 1, r) for r in range(20000)])
    assert stats.kstest(u, "uniform").pvalue > 1e-3


# ------------------------------------------------------------------ element decoding, reps

def test_bf16_decoding_matches_torch():
    bits = np.random.default_rng(0).integers(0, 2**16, size=4000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]           # finite values only
    got = oracle.elem_values(bits)
    want = _decoded(bits)
    assert np.array_equal(got, want)


def test_reps_are_means_of_valid_keys():
    """Representative = mean key of the team (explainer 三 step 2: the mean key), partial last
    team averaged over its valid keys only, an empty page gives zeros."""
    cfg = _tiny(dtype="bf16", batch=2, kv_heads=2, q_heads=4, seq_len=37, paged=True,
                num_pages=13)
    wl = W.generate(cfg, seq_lens=[37, 20], invalid_fill=float("nan"))
    reps = oracle.build_reps(_problem(wl), wl.page_fill)
    K = _decoded(wl.k_pool)
    for p in range(wl.num_pages):
        c = wl.page_fill[p]
        for h in range(cfg.kv_heads):
            want = K[p, h, :c].mean(axis=0) if c else np.zeros(cfg.head_dim)
            np.testing.assert_allclose(reps[p, h], want, rtol=1e-14, atol=1e-15)
    assert np.isfinite(reps).all()


# ------------------------------------------------------------------ team probabilities

def test_team_probs_equal_dense_attention_weights_for_single_token_teams():
    """With T = 1 the representative is the key, so each head's team softmax is that head's
    dense attention weight vector; p is their mean over the group.  Reference: torch SDPA
    in fp64 with V = identity (its output rows are the attention weights)."""
    cfg = _tiny(seq_len=50, team_size=1, head_dim=64, q_heads=4, kv_heads=2, batch=2)
    wl = W.generate(cfg)
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            K, _ = _unit_tokens(wl, b, h)
            q = torch.from_numpy(_decoded(wl.q[b, h * 2:(h + 1) * 2]))[None, :, None, :]
            k = torch.from_numpy(K)[None, None].expand(1, 2, -1, -1)
            eye = torch.eye(K.shape[0], dtype=torch.float64)[None, None].expand(1, 2, -1, -1)
            wts = torch.nn.functional.scaled_dot_product_attention(q, k, eye)[0, :, 0].numpy()
            p, s = oracle.team_probs(pr, reps, b, h, with_scores=True)
            np.testing.assert_allclose(p, wts.mean(axis=0), rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(s, _decoded(wl.q[b, h * 2:(h + 1) * 2]) @ K.T / 8.0,
                                       rtol=1e-12, atol=1e-13)


def test_team_probs_invariants():
    cfg = _tiny(seq_len=200, team_size=8, head_dim=16, q_heads=6, kv_heads=2)
    wl = W.generate(cfg)
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    p = oracle.team_probs(pr, reps, 0, 1)
    assert abs(p.sum() - 1.0) < 1e-14 and (p > 0).all()
    # a zero query scores every team alike: uniform distribution
    wl.q[:] = 0
    p0 = oracle.team_probs(_problem(wl), reps, 0, 1)
    np.testing.assert_allclose(p0, np.full(p0.size, 1.0 / p0.size), rtol=1e-15)


def test_team_probs_follow_the_page_table():
    """The same sequence stored contiguously or scattered over a permuted pool gives the same
    team distribution (teams are logical; pages are where they live)."""
    base = _tiny(seq_len=64, team_size=8, head_dim=16, q_heads=2, kv_heads=1, dtype="bf16")
    a = W.generate(base)
    b = W.generate(dataclasses.replace(base, paged=True, num_pages=20))
    assert not np.array_equal(a.page_table, b.page_table)
    pa, pb = _problem(a), _problem(b)
    np.testing.assert_array_equal(oracle.team_probs(pa, oracle.build_reps(pa), 0, 0),
                                  oracle.team_probs(pb, oracle.build_reps(pb), 0, 0))


# ------------------------------------------------------------------ sampling

def test_cdf_search_is_strict_and_skips_empty_teams():
    C = np.array([25, 25, 50, 100], dtype=np.uint64)   # team 1 has probability 0
    assert oracle.cdf_search(C, 0) == 0
    assert oracle.cdf_search(C, 24) == 0
    assert oracle.cdf_search(C, 25) == 2               # boundary belongs to the next team
    assert oracle.cdf_search(C, 75) == 3
    assert oracle.cdf_search(C, 100) == 3              # t >= Z: the completing team
    assert oracle.cdf_search(np.array([50, 100, 100], dtype=np.uint64), 100) == 1


def test_fixed_point_probabilities_round_half_away():
    assert oracle.fixed_prob(1.0) == 2**62
    assert oracle.fixed_prob(0.5) == 2**61
    assert oracle.fixed_prob(0.0) == 0
    assert oracle.fixed_prob(2.0**-63) == 1             # 0.5 rounds away from zero
    assert oracle.fixed_prob(2.0**-64) == 0             # 0.25 rounds to 0
    assert oracle.fixed_prob(3 * 2.0**-63) == 2         # 1.5 rounds to 2


def test_draws_are_exact_on_the_integer_cdf():
    """The draws equal an independent exact evaluation: Python integers for the fixed-point
    CDF and for floor(u Z) with u = (2x + 1) / 2^33, and bisect for the smallest team with
    t < C_i; the Philox words come from the pinned generator."""
    import bisect
    from fractions import Fraction
    rng = np.random.default_rng(3)
    for n, seed, b, h in [(7, 5, 0, 0), (64, 2**40 + 3, 3, 2), (300, 11, 1, 5)]:
        p = rng.dirichlet(np.full(n, 0.3))
        p[rng.integers(0, n)] = 0.0
        P = [int(Fraction(float(x)) * 2**62 + Fraction(1, 2)) for x in p]
        C = list(__import__("itertools").accumulate(P))
        Z = C[-1]
        M = 500
        draws, t, Co = oracle.draw(p, M, seed, b, h)
        assert [int(c) for c in Co] == C
        for r in range(M):
            x = int(oracle.philox4x32_10([r, h, b, 0], [seed & 0xFFFFFFFF, seed >> 32])[0])
            tr = ((2 * x + 1) * Z) >> 33
            assert int(t[r]) == tr
            assert draws[r] == bisect.bisect_right(C, tr)


def test_draws_follow_the_plain_definition_on_the_unrounded_probabilities():
    """The fixed-point draws against the method's plain definition, taken exactly: with the
    fp64 probabilities p as exact rationals, C_i = p_0 + ... + p_i, Z = C_{n-1} and
    u = (x + 1/2) / 2^32 (x the draw's Philox word), draw r is the smallest i with
    u Z < C_i (M teams drawn according to p, explainer section 三 step 3).  The
    62-bit rounding of p may move a draw only across a boundary that u Z lies within
    1e-12 Z of; such draws are counted and must be rare, every other draw must agree."""
    import bisect
    from fractions import Fraction
    rng = np.random.default_rng(17)
    near, total = 0, 0
    for n, M, seed, b, h in [(5, 400, 9, 0, 0), (64, 800, 2**33 + 1, 2, 1),
                             (256, 1000, 31, 0, 3), (1024, 600, 123456789, 5, 0)]:
        p = rng.dirichlet(np.full(n, 0.5))
        p[rng.integers(0, n, size=max(1, n // 16))] = 0.0          # empty teams
        p[rng.integers(0, n)] = 1e-300                              # far below 2^-62
        C, acc = [], Fraction(0)
        for x in p:
            acc += Fraction(float(x))
            C.append(acc)
        Z = C[-1]
        draws, _, _ = oracle.draw(p, M, seed, b, h)
        for r in range(M):
            x = int(oracle.philox4x32_10([r, h, b, 0], [seed & 0xFFFFFFFF, seed >> 32])[0])
            uZ = Fraction(2 * x + 1, 2**33) * Z
            plain = bisect.bisect_right(C, uZ)        # smallest i with uZ < C_i
            total += 1
            if draws[r] != plain:
                lo, hi = sorted((int(draws[r]), plain))
                gap = min(abs(uZ - C[i]) for i in range(lo, hi))
                assert gap <= Fraction(1, 10**12) * Z, (n, r, draws[r], plain, float(gap / Z))
                near += 1
            assert p[draws[r]] > 0.0                  # an empty team is never drawn
    assert near <= 1e-4 * total, (near, total)


def test_draw_frequencies_follow_p():
    """Chi-square goodness of fit of 200000 draws to p; a zero-probability team is never
    drawn (an off-by-one in the inverse CDF shifts mass and fails this)."""
    from scipy import stats
    p = np.array([0.05, 0.3, 0.0, 0.15, 0.4, 0.1])
    draws, t, C = oracle.draw(p, 200000, seed=77, b=0, h=0)
    counts = np.bincount(draws, minlength=p.size)
    assert counts[2] == 0
    nz = p > 0
    assert stats.chisquare(counts[nz], p[nz] * draws.size).pvalue > 1e-4
    np.testing.assert_allclose(C.astype(np.float64) / 2.0**62, np.cumsum(p), rtol=0, atol=1e-15)


def test_inclusion_probability_golden():
    rows = np.loadtxt(os.path.join(GOLDEN, "inclusion_probability.txt"))
    for p, M, pi in rows:
        M = int(M)
        _, got = oracle.select(np.zeros(M, np.int32), np.array([p, 1.0 - p]))
        assert abs(got[0] - pi) <= 1e-15, (p, M, got[0], pi)


@pytest.mark.parametrize("n,M", [(3, 1), (4, 3), (5, 4), (2, 6)])
def test_inclusion_probability_matches_enumeration(n, M):
    p = np.random.default_rng(n * 10 + M).dirichlet(np.ones(n))
    incl = np.zeros(n)
    for seq in itertools.product(range(n), repeat=M):
        prob = np.prod(p[list(seq)])
        for i in set(seq):
            incl[i] += prob
    # pi_i depends only on p_i and M: ask for it with M draws that all hit team i
    for i in range(n):
        _, pii = oracle.select(np.full(M, i, np.int32), p)
        assert abs(pii[0] - incl[i]) <= 1e-14, (i, pii[0], incl[i])


# ------------------------------------------------------------------ the estimator

def _read_golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = np.array([float(x) for x in v.split()])
    return vals


def _two_team_problem(g):
    q = np.array([[[g["q"][0]]]], np.float32)
    k = np.array(g["k"], np.float32).reshape(2, 1, 1, 1)
    v = np.array(g["v"], np.float32).reshape(2, 1, 1, 1)
    return oracle.Problem(q, k, v, np.array([[0, 1]], np.int32), np.array([2], np.int32))


def test_worked_two_team_example():
    """Hand-derived worked example (tests/golden/worked_two_teams.txt): team probabilities,
    inclusion probabilities, per-outcome estimates and exact expectations."""
    g = _read_golden("worked_two_teams.txt")
    pr = _two_team_problem(g)
    reps = oracle.build_reps(pr)
    p = oracle.team_probs(pr, reps, 0, 0)
    np.testing.assert_allclose(p, g["p"], rtol=1e-7)
    M = int(g["M"][0])
    pi = np.array([oracle.select(np.full(M, i, np.int32), p)[1][0] for i in range(2)])
    np.testing.assert_allclose(pi, g["pi"], rtol=1e-7)
    out = {}
    for S in [(0,), (1,), (0, 1)]:
        out[S] = oracle.attend(pr, 0, 0, np.array(S, np.int32), pi[list(S)])[0, 0]
    np.testing.assert_allclose([out[(0,)], out[(1,)], out[(0, 1)]],
                               [g["out_S0"][0], g["out_S1"][0], g["out_S01"][0]], rtol=1e-7)
    E_num = E_den = E_out = 0.0
    for seq in itertools.product(range(2), repeat=M):
        prob = np.prod(p[list(seq)])
        S = tuple(sorted(set(seq)))
        num, den = oracle.num_den(pr, 0, 0, np.array(S, np.int32), pi[list(S)], 0.0)
        E_num += prob * num[0, 0]
        E_den += prob * den[0]
        E_out += prob * out[S]
    np.testing.assert_allclose([E_num, E_den, E_out],
                               [g["E_num"][0], g["E_den"][0], g["E_out"][0]], rtol=1e-6)
    np.testing.assert_allclose(oracle.dense(pr, 0, 0)[0, 0], g["dense"][0], rtol=1e-7)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_expectation_by_enumeration_equals_dense_sums(M):
    """E[num] and E[den] over all n^M ordered draw sequences equal the dense sums
    sum_j e^{s_j - m} v_j and sum_j e^{s_j - m} (importance-sampling correction, explainer
    3.1; "estimates attention over the full cache", abstract).  Partial last team, G = 2."""
    cfg = _tiny(seq_len=19, team_size=4, head_dim=4, q_heads=2, kv_heads=1, data_seed=3)
    wl = W.generate(cfg, invalid_fill=float("nan"))
    pr = _problem(wl)
    reps = oracle.build_reps(pr, wl.page_fill)
    p = oracle.team_probs(pr, reps, 0, 0)
    n = p.size
    assert n == 5
    shift = np.array([0.3, -0.2])
    E_num = np.zeros((2, cfg.head_dim))
    E_den = np.zeros(2)
    for seq in itertools.product(range(n), repeat=M):
        prob = np.prod(p[list(seq)])
        sel, pi = oracle.select(np.array(seq, np.int32), p)
        num, den = oracle.num_den(pr, 0, 0, sel, pi, shift)
        E_num += prob * num
        E_den += prob * den
    K, V = _unit_tokens(wl, 0, 0)
    q = _decoded(wl.q[0])
    e = np.exp(q @ K.T / np.sqrt(cfg.head_dim) - shift[:, None])
    np.testing.assert_allclose(E_den, e.sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(E_num, e @ V, rtol=1e-12, atol=1e-12)


def test_dense_special_case_all_pi_one():
    """With M so large that every pi_i == 1.0 in fp64 and every team drawn, the estimate is
    dense softmax attention: checked against brute force and torch SDPA (fp64)."""
    wl = W.generate("tiny_f32")
    wl.q[:] = wl.q * np.float32(0.05)                  # near-uniform team distribution
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    M = 4096
    r = oracle.decode(pr, reps, M, 9, 0, 0)
    assert r.sel.size == wl.cfg.n_teams and (r.pi == 1.0).all()
    dense_np = _dense_numpy(wl, 0, 0)
    np.testing.assert_allclose(r.out, dense_np, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.dense(pr, 0, 0), dense_np, rtol=0, atol=1e-12)
    K, V = _unit_tokens(wl, 0, 0)
    q = torch.from_numpy(_decoded(wl.q[0]))[None, :, None, :]
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        q, torch.from_numpy(K)[None, None].expand(1, 2, -1, -1),
        torch.from_numpy(V)[None, None].expand(1, 2, -1, -1))[0, :, 0].numpy()
    np.testing.assert_allclose(r.out, sdpa, rtol=0, atol=1e-12)


def test_dense_special_case_every_kv_head():
    """The all-pi-one case on every unit of a multi-head, multi-sequence, paged problem:
    2 sequences of different lengths (partial last teams), 3 KV heads with G = 2, a permuted
    page pool.  Each unit's estimate and the oracle's dense attention equal textbook softmax
    attention over that unit's own keys and values (numpy, fp64)."""
    cfg = _tiny(batch=2, q_heads=6, kv_heads=3, head_dim=8, team_size=8, paged=True,
                num_pages=16, data_seed=21)
    wl = W.generate(cfg, seq_lens=[37, 21], invalid_fill=float("nan"))
    wl.q[:] = wl.q * np.float32(0.05)                  # near-uniform team distribution
    pr = _problem(wl)
    reps = oracle.build_reps(pr, wl.page_fill)
    for b in range(2):
        for h in range(3):
            r = oracle.decode(pr, reps, 4096, 3, b, h)
            assert r.sel.size == -(-int(wl.seq_lens[b]) // 8) and (r.pi == 1.0).all()
            want = _dense_numpy(wl, b, h)
            np.testing.assert_allclose(r.out, want, rtol=0, atol=1e-12)
            np.testing.assert_allclose(oracle.dense(pr, b, h), want, rtol=0, atol=1e-12)


def test_single_team_sequence_is_exact():
    cfg = _tiny(seq_len=6, team_size=8, head_dim=8)
    wl = W.generate(cfg, invalid_fill=float("nan"))
    pr = _problem(wl)
    r = oracle.decode(pr, oracle.build_reps(pr, wl.page_fill), 5, 1, 0, 0)
    assert list(r.sel) == [0] and r.pi[0] == 1.0 and (r.draws == 0).all()
    np.testing.assert_allclose(r.out, _dense_numpy(wl, 0, 0), atol=1e-13)


def test_monte_carlo_unbiased_num_and_den():
    """Over 4096 seeds of the tiny fp32 workload (M = 8), the means of the HT denominator
    and of <numerator, w> lie within 3 standard errors of the dense values."""
    wl = W.generate("tiny_f32")
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    p = oracle.team_probs(pr, reps, 0, 0)
    K, V = _unit_tokens(wl, 0, 0)
    q = _decoded(wl.q[0])
    s = q @ K.T / 8.0
    shift = s.max(axis=1)
    e = np.exp(s - shift[:, None])
    dense_den, dense_num = e.sum(axis=1), e @ V
    w = np.random.default_rng(0).standard_normal(64)
    w /= np.linalg.norm(w)
    dens, nums, ratios = [], [], []
    for seed in range(4096):
        draws, _, _ = oracle.draw(p, 8, seed, 0, 0)
        sel, pi = oracle.select(draws, p)
        num, den = oracle.num_den(pr, 0, 0, sel, pi, shift)
        dens.append(den)
        nums.append(num @ w)
    dens, nums = np.array(dens), np.array(nums)
    for est, truth in [(dens, dense_den), (nums, dense_num @ w)]:
        se = est.std(axis=0, ddof=1) / np.sqrt(est.shape[0])
        assert (np.abs(est.mean(axis=0) - truth) < 3 * se).all(), (est.mean(axis=0), truth, se)


def test_decode_chains_the_steps():
    wl = W.generate(_tiny(seq_len=100, team_size=8, head_dim=16, q_heads=4, kv_heads=2,
                          dtype="bf16"))
    pr = _problem(wl)
    reps = oracle.build_reps(pr)
    for h in range(2):
        r = oracle.decode(pr, reps, 6, 42, 0, h)
        p = oracle.team_probs(pr, reps, 0, h)
        draws, _, _ = oracle.draw(p, 6, 42, 0, h)
        sel, pi = oracle.select(draws, p)
        assert np.array_equal(r.draws, draws) and np.array_equal(r.sel, sel)
        np.testing.assert_array_equal(r.out, oracle.attend(pr, 0, h, sel, pi))


def test_invalid_slots_never_reach_the_output():
    """Page slots past the end of a sequence hold NaN; nothing of them leaks into reps,
    probabilities or the estimate."""
    cfg = _tiny(seq_len=45, team_size=8, head_dim=8)
    a = W.generate(cfg, invalid_fill=float("nan"))
    b = W.generate(cfg, invalid_fill=0.0)
    ra = oracle.decode(_problem(a), oracle.build_reps(_problem(a), a.page_fill), 4, 3, 0, 0)
    rb = oracle.decode(_problem(b), oracle.build_reps(_problem(b), b.page_fill), 4, 3, 0, 0)
    assert np.isfinite(ra.out).all()
    np.testing.assert_array_equal(ra.out, rb.out)
