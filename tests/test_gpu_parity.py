"""GPU parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Rules: sampled team ids bit-exact, except draws whose oracle u*Z lies within 1e-6 of an
oracle CDF value (counted, < 1e-4 of draws); inclusion probabilities within 1e-5 relative;
outputs computed on identical sampled sets (the oracle's) within 1e-5 max-abs for fp32
inputs and 2e-3 for bf16 inputs; representatives and dense attention likewise.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import sampled_sparse_decode_gb300 as santa
from sampled_sparse_decode_gb300 import workloads as W
from helpers import (BOUNDARY_SHARE, TOL_OUT, TOL_PI, DeviceWorkload, compare_draws,
                     full_oracle_reps, full_workload, problem)

pytestmark = pytest.mark.gpu

NAN = float("nan")

# Reduced-size variants of every workload: the same distributions, several tiles per unit,
# ragged sequence ends (NaN in the unused page slots) and mixed lengths in one batch.
SMALL = {
    "tiny_f32": dict(cfg="tiny_f32"),
    "qwen_b2_ragged": dict(cfg="qwen7b_32k_b1_m31", batch=2, seq_len=4000),
    "qwen_b3_mixed_m64": dict(cfg="qwen7b_32k_b8_m64", batch=3, seq_lens=[4096, 3000, 129]),
    "llama_paged_b4": dict(cfg="llama8b_paged_32k_b16_m32", batch=4, seq_len=6000,
                           num_pages=300),
    "long_paged_b2": dict(cfg="long_128k_b4_m64", batch=2, seq_len=20000, num_pages=0),
    "bf16_d64_t64": dict(cfg="qwen7b_32k_b1_m31", head_dim=64, team_size=64, seq_len=3000,
                         q_heads=8, kv_heads=2, draws=20),
    "f32_d128_g8": dict(cfg="tiny_f32", head_dim=128, team_size=128, seq_len=5000,
                        q_heads=16, kv_heads=2, draws=12),
    # one long sequence, one KV head: dense work spans several clusters
    "long_b1_multicluster": dict(cfg="long_128k_b4_m64", batch=1, q_heads=7, kv_heads=1,
                                 seq_len=40000, draws=600, num_pages=0),
    # 160 units: more CTAs than SMs, so bf16 steps take the two-CTA-per-SM variant (the
    # smaller cases take the wide one-CTA-per-SM variant)
    "qwen_b40_two_per_sm": dict(cfg="qwen7b_32k_b8_m64", batch=40, seq_len=1300),
    # 4096 draws over 4096 teams: more chunks than one cluster's tables hold, so the sampled
    # step itself spans two clusters (partials through the workspace)
    "f32_b1_two_clusters": dict(cfg="tiny_f32", seq_len=4096 * 128, team_size=128,
                                draws=4096),
}


def test_multicluster_cases_take_the_multicluster_path():
    for name, which in [("long_b1_multicluster", "dense"), ("f32_b1_two_clusters", "decode"),
                        ("f32_b1_two_clusters", "attend")]:
        wl = make(SMALL[name])
        dw = DeviceWorkload(wl)
        plan = santa.santa_decode_plan(dw.q, dw.k_pool, dw.page_table, wl.cfg.draws, which)
        assert plan["clusters_per_unit"] >= 2, (name, which, plan)


def test_both_kernel_variants_are_covered():
    for name, want in [("qwen_b2_ragged", True), ("bf16_d64_t64", True),
                       ("qwen_b40_two_per_sm", False)]:
        wl = make(SMALL[name])
        dw = DeviceWorkload(wl)
        for which in ("decode", "attend", "dense"):
            plan = santa.santa_decode_plan(dw.q, dw.k_pool, dw.page_table, wl.cfg.draws, which)
            assert plan["wide"] == want, (name, which, plan)
        assert not santa.santa_decode_plan(dw.q, dw.k_pool, dw.page_table, wl.cfg.draws,
                                           "sample")["wide"]


def test_compact_and_general_forms_are_both_covered():
    """bf16 decode steps run the compact form of the kernel (both variants, every sampler and
    the mixture; bf16 sampling-only steps too); fp32 steps and units spread over several
    clusters run the general form, and so do the attention-only and dense modes.  The parity
    tests below cover each."""
    cases = [("qwen_b2_ragged", {}, "compact"), ("bf16_d64_t64", {}, "compact"),
             ("qwen_b40_two_per_sm", {}, "compact"), ("llama_paged_b4", {}, "compact"),
             ("long_paged_b2", {}, "compact"), ("qwen_b3_mixed_m64", {}, "compact"),
             ("long_b1_multicluster", {}, "compact"),
             ("tiny_f32", {}, "general"), ("f32_d128_g8", {}, "general"),
             ("f32_b1_two_clusters", {}, "general"),
             ("qwen_b2_ragged", dict(sampler="systematic"), "compact"),
             ("qwen_b2_ragged", dict(sampler="iid_hh"), "compact"),
             ("qwen_b2_ragged", dict(mix_alpha=0.05), "compact")]
    for name, kw, want in cases:
        wl = make(SMALL[name])
        dw = DeviceWorkload(wl)
        got = santa.santa_decode_path(dw.q, dw.k_pool, dw.page_table, wl.cfg.draws, **kw)
        assert got == want, (name, kw, got)
    for name in FULL:
        wl = full_workload(name)
        dw = DeviceWorkload(wl)
        assert santa.santa_decode_path(dw.q, dw.k_pool, dw.page_table, wl.cfg.draws) == \
            "compact", name


def make(spec, **extra):
    spec = dict(spec, **extra)
    name = spec.pop("cfg")
    seq_lens = spec.pop("seq_lens", None)
    if seq_lens is not None:
        spec["batch"] = len(seq_lens)
    return W.generate(name, seq_lens=seq_lens, invalid_fill=NAN, **spec)


def run_sample(dw: DeviceWorkload, reps, M, seed):
    bufs = santa.santa_sample(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                              M, seed, team_probs=True)
    torch.cuda.synchronize()
    return bufs


def check_unit_sampling(wl, pr, reps_o, bufs, M, seed, b, h):
    """Compares one unit's p, draws, S and pi with the oracle; returns draw statistics."""
    p = oracle.team_probs(pr, reps_o, b, h)
    n = p.size
    p_gpu = bufs.team_probs[b, h, :n].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(p_gpu, p, rtol=1e-5, atol=1e-7 * p.max())
    assert (bufs.team_probs[b, h, n:].cpu().numpy() == 0).all()
    draws, t, C = oracle.draw(p, M, seed, b, h)
    g_draws = bufs.draw_ids[b, h].cpu().numpy()
    inside, outside = compare_draws(g_draws, draws, t, C)
    assert outside == 0, f"unit ({b},{h}): {outside} draws differ away from any CDF boundary"
    cnt = int(bufs.sel_count[b, h])
    sel = bufs.sel_ids[b, h].cpu().numpy()
    pi = bufs.pi[b, h].cpu().numpy()
    # S is the ascending distinct set of the GPU's own draws, padded with -1 / 0
    assert np.array_equal(sel[:cnt], np.unique(g_draws))
    assert (sel[cnt:] == -1).all() and (pi[cnt:] == 0).all()
    if inside == 0:
        o_sel, o_pi = oracle.select(draws, p)
        assert np.array_equal(sel[:cnt], o_sel)
        np.testing.assert_allclose(pi[:cnt], o_pi, rtol=TOL_PI)
    return inside, M


def check_unit_attend(wl, pr, dw, b, h, o_sel, o_pi, out_gpu, tol):
    want = oracle.attend(pr, b, h, o_sel, o_pi)
    G = wl.cfg.group
    got = out_gpu[b, h * G:(h + 1) * G].cpu().numpy().astype(np.float64)
    err = np.abs(got - want).max()
    assert err <= tol, f"unit ({b},{h}): max-abs error {err:.3g} > {tol}"
    return err


@pytest.mark.parametrize("name", list(SMALL))
def test_reps_parity(name):
    wl = make(SMALL[name])
    dw = DeviceWorkload(wl)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    torch.cuda.synchronize()
    want = oracle.build_reps(problem(wl), wl.page_fill)
    got = reps.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max())


@pytest.mark.parametrize("name", list(SMALL))
def test_sample_and_attend_parity(name):
    wl = make(SMALL[name])
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr, wl.page_fill)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    seed = 1234
    bufs = run_sample(dw, reps, cfg.draws, seed)
    inside = total = 0
    sels, pis, units = [], [], []
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            i, m = check_unit_sampling(wl, pr, reps_o, bufs, cfg.draws, seed, b, h)
            inside, total = inside + i, total + m
            p = oracle.team_probs(pr, reps_o, b, h)
            d, _, _ = oracle.draw(p, cfg.draws, seed, b, h)
            s, pi = oracle.select(d, p)
            units.append((b, h))
            sels.append(s)
            pis.append(pi)
    assert inside <= BOUNDARY_SHARE * total
    # attention on the oracle's sampled sets and inclusion probabilities
    M = cfg.draws
    sel_t = torch.full((cfg.batch, cfg.kv_heads, M), -1, dtype=torch.int32)
    cnt_t = torch.zeros((cfg.batch, cfg.kv_heads), dtype=torch.int32)
    pi_t = torch.zeros((cfg.batch, cfg.kv_heads, M), dtype=torch.float32)
    for (b, h), s, pi in zip(units, sels, pis):
        sel_t[b, h, :s.size] = torch.from_numpy(s)
        cnt_t[b, h] = s.size
        pi_t[b, h, :s.size] = torch.from_numpy(pi.astype(np.float32))
    ab = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens,
                            sel_t.cuda(), cnt_t.cuda(), pi_t.cuda())
    torch.cuda.synchronize()
    assert ab.status() == 0
    tol = TOL_OUT[cfg.dtype]
    for (b, h), s, pi in zip(units, sels, pis):
        check_unit_attend(wl, pr, dw, b, h, s, pi, ab.out, tol)
    # the whole step in one call: same sets wherever the draws agreed
    db = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                            seed)
    torch.cuda.synchronize()
    assert db.status() == 0
    for (b, h), s, pi in zip(units, sels, pis):
        if int(db.sel_count[b, h]) == s.size and np.array_equal(
                db.sel_ids[b, h, :s.size].cpu().numpy(), s):
            check_unit_attend(wl, pr, dw, b, h, s, pi, db.out, tol)


@pytest.mark.parametrize("name", list(SMALL))
def test_dense_parity(name):
    wl = make(SMALL[name])
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    bufs = santa.santa_dense_decode(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens)
    torch.cuda.synchronize()
    assert bufs.status() == 0
    G, tol = wl.cfg.group, TOL_OUT[wl.cfg.dtype]
    for b in range(wl.cfg.batch):
        for h in range(wl.cfg.kv_heads):
            want = oracle.dense(pr, b, h)
            got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
            assert np.abs(got - want).max() <= tol


def test_seed_sweep_draws_bit_exact():
    """4096 decode seeds of the tiny fp32 workload: every draw equals the oracle's, except
    draws inside the CDF-boundary window, which stay below 1e-4 of all draws."""
    wl = W.generate("tiny_f32")
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr)
    reps = santa.santa_build_reps(dw.k_pool)
    p = oracle.team_probs(pr, reps_o, 0, 0)
    M = wl.cfg.draws
    bufs = None
    seeds = range(4096)
    gpu = torch.empty((len(seeds), M), dtype=torch.int32, device="cuda")
    for k, seed in enumerate(seeds):
        bufs = santa.santa_sample(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                                  M, seed, bufs=bufs)
        gpu[k].copy_(bufs.draw_ids[0, 0])
    gpu = gpu.cpu().numpy()
    inside = 0
    for k, seed in enumerate(seeds):
        draws, t, C = oracle.draw(p, M, seed, 0, 0)
        i, o = compare_draws(gpu[k], draws, t, C)
        assert o == 0, f"seed {seed}: draws differ away from a CDF boundary"
        inside += i
    assert inside < BOUNDARY_SHARE * gpu.size


FULL = ["qwen7b_32k_b1_m31", "qwen7b_32k_b8_m64", "llama8b_paged_32k_b16_m32", "long_128k_b4_m64"]


def spread_units(batch, kv_heads, n=8):
    """Up to n (sequence, KV head) units spread evenly over the batch and the heads."""
    idx = np.unique(np.linspace(0, batch * kv_heads - 1, min(n, batch * kv_heads)).round())
    return [(int(i) // kv_heads, int(i) % kv_heads) for i in idx]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_units(name):
    """Full-size workloads in the launch configuration the benchmark times (santa_decode and
    santa_attend with the default workspace).  On up to 8 units spread over the batch and
    the heads, the oracle checks p, the draws, S and pi; santa_attend is then fed the
    oracle's own S and pi for those units (the GPU's for the others, so the launch is the
    full one) and its outputs are compared with the oracle's on the same sets; the fused
    step's outputs are compared wherever its sets equal the oracle's (at least one unit)."""
    wl = full_workload(name)
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = full_oracle_reps(name)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    seed = 7
    bufs = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                              cfg.draws, seed, team_probs=True)
    torch.cuda.synchronize()
    assert bufs.status() == 0
    units = spread_units(cfg.batch, cfg.kv_heads)
    assert len(units) == min(8, cfg.batch * cfg.kv_heads)
    tol = TOL_OUT[cfg.dtype]
    sel_t, cnt_t, pi_t = bufs.sel_ids.clone(), bufs.sel_count.clone(), bufs.pi.clone()
    oracle_sets = {}
    fused_checked = 0
    for b, h in units:
        check_unit_sampling(wl, pr, reps_o, bufs, cfg.draws, seed, b, h)
        p = oracle.team_probs(pr, reps_o, b, h)
        d, _, _ = oracle.draw(p, cfg.draws, seed, b, h)
        s, pi = oracle.select(d, p)
        oracle_sets[(b, h)] = (s, pi)
        sel_t[b, h] = -1
        sel_t[b, h, :s.size] = torch.from_numpy(s).cuda()
        cnt_t[b, h] = s.size
        pi_t[b, h] = 0.0
        pi_t[b, h, :s.size] = torch.from_numpy(pi.astype(np.float32)).cuda()
        if int(bufs.sel_count[b, h]) == s.size and np.array_equal(
                bufs.sel_ids[b, h, :s.size].cpu().numpy(), s):
            check_unit_attend(wl, pr, dw, b, h, s, pi, bufs.out, tol)
            fused_checked += 1
    assert fused_checked >= 1
    ab = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, sel_t,
                            cnt_t, pi_t)
    torch.cuda.synchronize()
    assert ab.status() == 0
    for (b, h), (s, pi) in oracle_sets.items():
        check_unit_attend(wl, pr, dw, b, h, s, pi, ab.out, tol)
    # properties that hold for every unit at any size
    cnt = bufs.sel_count.cpu().numpy()
    assert (cnt >= 1).all() and (cnt <= min(cfg.draws, cfg.n_teams)).all()
    assert torch.isfinite(bufs.out).all()
    pi = bufs.pi.cpu().numpy()
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            assert (pi[b, h, :cnt[b, h]] > 0).all() and (pi[b, h, :cnt[b, h]] <= 1).all()


@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 8])
@pytest.mark.parametrize("head_dim,batch", [(128, 2), (64, 1), (128, 40)])
def test_every_group_size(G, head_dim, batch):
    """Every instantiated group size, both head sizes; batch 40 takes the two-CTA-per-SM
    variant, the others the wide one.  Draws, S and pi as in the sampling parity test; the
    whole step compared with the oracle where the sampled sets agree."""
    wl = make(dict(cfg="qwen7b_32k_b1_m31", batch=batch, q_heads=2 * G, kv_heads=2,
                   head_dim=head_dim, seq_len=1100 if batch > 2 else 2600, draws=24))
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr, wl.page_fill)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    want_wide = batch <= 2
    plan = santa.santa_decode_plan(dw.q, dw.k_pool, dw.page_table, cfg.draws, "decode")
    assert plan["wide"] == want_wide, plan
    bufs = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                              cfg.draws, 31, team_probs=True)
    torch.cuda.synchronize()
    assert bufs.status() == 0
    tol = TOL_OUT[cfg.dtype]
    checked = 0
    for b in range(0, cfg.batch, max(1, cfg.batch // 4)):
        for h in range(cfg.kv_heads):
            check_unit_sampling(wl, pr, reps_o, bufs, cfg.draws, 31, b, h)
            r = oracle.decode(pr, reps_o, cfg.draws, 31, b, h)
            cnt = int(bufs.sel_count[b, h])
            if cnt == r.sel.size and np.array_equal(bufs.sel_ids[b, h, :cnt].cpu().numpy(), r.sel):
                got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
                assert np.abs(got - r.out).max() <= tol
                checked += 1
    assert checked >= 1
