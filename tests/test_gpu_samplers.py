"""GPU parity of the sampler variants (systematic draws, Hansen-Hurwitz weights, defensive
uniform mixture) against the oracle, through the C ABI.

Same rules as the plain method: sampled team ids bit-exact except draws whose oracle point
lies within the CDF-boundary window (counted, < 1e-4 of draws); 1 / weight per team within
1e-5 relative; the sampling distribution q within 1e-5 relative; outputs on identical
sampled sets within 1e-5 (fp32) / 2e-3 (bf16) max-abs.
"""
import numpy as np
import pytest
import torch

import oracle
import sampled_sparse_decode_gb300 as santa
from helpers import BOUNDARY_SHARE, TOL_OUT, TOL_PI, DeviceWorkload, compare_draws, problem
from test_gpu_parity import SMALL, make

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny_f32", "systematic", 0.0),
    ("tiny_f32", "iid_hh", 0.0),
    ("qwen_b2_ragged", "systematic", 0.05),
    ("qwen_b2_ragged", "iid_hh", 0.1),
    ("llama_paged_b4", "iid_ht", 0.1),
    ("llama_paged_b4", "systematic", 0.0),
    ("bf16_d64_t64", "iid_hh", 0.02),
    ("qwen_b40_two_per_sm", "systematic", 0.1),
]


@pytest.mark.parametrize("name,sampler,alpha", CASES)
def test_sampler_parity(name, sampler, alpha):
    wl = make(SMALL[name])
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr, wl.page_fill)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    M, seed = cfg.draws, 4321
    bufs = santa.santa_sample(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                              seed, team_probs=True, sampler=sampler, mix_alpha=alpha)
    torch.cuda.synchronize()
    assert bufs.status() == 0
    inside = total = 0
    units = []
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            q = oracle.mix(oracle.team_probs(pr, reps_o, b, h), alpha)
            n = q.size
            q_gpu = bufs.team_probs[b, h, :n].cpu().numpy().astype(np.float64)
            np.testing.assert_allclose(q_gpu, q, rtol=1e-5, atol=1e-7 * q.max())
            draws, t, C = oracle.draw_with(sampler, q, M, seed, b, h)
            g_draws = bufs.draw_ids[b, h].cpu().numpy()
            i, o = compare_draws(g_draws, draws, t, C)
            assert o == 0, f"unit ({b},{h}): {o} draws differ outside the boundary window"
            inside, total = inside + i, total + M
            sel, rc = oracle.select_ex(draws, q, sampler)
            cnt = int(bufs.sel_count[b, h])
            g_sel = bufs.sel_ids[b, h].cpu().numpy()
            g_rc = bufs.pi[b, h].cpu().numpy().astype(np.float64)
            assert (g_sel[cnt:] == -1).all() and (g_rc[cnt:] == 0).all()
            if np.array_equal(g_draws, draws):
                assert np.array_equal(g_sel[:cnt], sel)
                np.testing.assert_allclose(g_rc[:cnt], rc, rtol=TOL_PI)
            units.append(((b, h), sel, rc))
    assert inside <= BOUNDARY_SHARE * total
    # attention on the oracle's sets with the oracle's weights, and the whole step
    sel_t = torch.full((cfg.batch, cfg.kv_heads, M), -1, dtype=torch.int32)
    cnt_t = torch.zeros((cfg.batch, cfg.kv_heads), dtype=torch.int32)
    rc_t = torch.zeros((cfg.batch, cfg.kv_heads, M), dtype=torch.float32)
    for (b, h), sel, rc in units:
        sel_t[b, h, :sel.size] = torch.from_numpy(sel)
        cnt_t[b, h] = sel.size
        rc_t[b, h, :sel.size] = torch.from_numpy(rc.astype(np.float32))
    ab = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens,
                            sel_t.cuda(), cnt_t.cuda(), rc_t.cuda())
    db = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                            seed, sampler=sampler, mix_alpha=alpha)
    torch.cuda.synchronize()
    assert ab.status() == 0 and db.status() == 0
    G, tol = cfg.group, TOL_OUT[cfg.dtype]
    for (b, h), sel, rc in units:
        want = oracle.attend(pr, b, h, sel, rc)
        got = ab.out[b, h * G:(h + 1) * G].cpu().numpy()
        assert np.abs(got - want).max() <= tol
        if int(db.sel_count[b, h]) == sel.size and np.array_equal(
                db.sel_ids[b, h, :sel.size].cpu().numpy(), sel):
            got = db.out[b, h * G:(h + 1) * G].cpu().numpy()
            assert np.abs(got - want).max() <= tol


def test_decode_ex_end_to_end_matches_oracle_unit():
    """santa_decode with a variant against the oracle's whole step for one unit."""
    wl = make(SMALL["qwen_b3_mixed_m64"])
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr, wl.page_fill)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    for sampler, alpha in [("systematic", 0.1), ("iid_hh", 0.0)]:
        db = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                                wl.cfg.draws, 99, sampler=sampler, mix_alpha=alpha)
        torch.cuda.synchronize()
        for b in range(wl.cfg.batch):
            r = oracle.decode_ex(pr, reps_o, wl.cfg.draws, 99, b, 1, sampler, alpha)
            cnt = int(db.sel_count[b, 1])
            if cnt == r.sel.size and np.array_equal(db.sel_ids[b, 1, :cnt].cpu().numpy(), r.sel):
                G = wl.cfg.group
                got = db.out[b, G:2 * G].cpu().numpy()
                assert np.abs(got - r.out).max() <= TOL_OUT[wl.cfg.dtype]


def test_variants_reject_shapes_sampled_across_ctas():
    """More teams per unit than one CTA samples (4096 > 1024): variants are refused."""
    wl = make(SMALL["f32_b1_two_clusters"])
    dw = DeviceWorkload(wl)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    for sampler, alpha in [("systematic", 0.0), ("iid_ht", 0.1)]:
        with pytest.raises(santa.SantaError, match="unsupported"):
            santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                               wl.cfg.draws, 1, sampler=sampler, mix_alpha=alpha)
    # the plain method still runs there
    santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                       wl.cfg.draws, 1)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,sampler,alpha", [
    ("qwen7b_32k_b1_m31", "systematic", 0.05),
    ("qwen7b_32k_b8_m64", "iid_hh", 0.0),
    ("llama8b_paged_32k_b16_m32", "iid_ht", 0.05),
    ("long_128k_b4_m64", "systematic", 0.0),
])
def test_sampler_variants_at_full_size(name, sampler, alpha):
    """The sampler variants on the full-size workloads, in the launch shape the accuracy
    benchmark uses (the compact form's variant instantiations).  On up to 8 units spread over
    the batch and the heads: q, the draws (window rule), S and 1 / weight against the oracle;
    then santa_attend on the oracle's sets and weights for those units against the oracle's
    attention, and the whole step's outputs wherever its sets equal the oracle's."""
    from helpers import full_oracle_reps, full_workload
    from test_gpu_parity import spread_units
    wl = full_workload(name)
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = full_oracle_reps(name)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    M, seed = cfg.draws, 2024
    assert santa.santa_decode_path(dw.q, dw.k_pool, dw.page_table, M, sampler=sampler,
                                   mix_alpha=alpha) == "compact"
    bufs = santa.santa_sample(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                              seed, team_probs=True, sampler=sampler, mix_alpha=alpha)
    db = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                            seed, sampler=sampler, mix_alpha=alpha)
    torch.cuda.synchronize()
    assert bufs.status() == 0 and db.status() == 0
    # the whole step draws exactly what the sampling-only launch draws
    assert torch.equal(db.draw_ids, bufs.draw_ids) and torch.equal(db.sel_count, bufs.sel_count)
    inside = total = 0
    sel_t, cnt_t, rc_t = bufs.sel_ids.clone(), bufs.sel_count.clone(), bufs.pi.clone()
    units = []
    for b, h in spread_units(cfg.batch, cfg.kv_heads):
        q = oracle.mix(oracle.team_probs(pr, reps_o, b, h), alpha)
        n = q.size
        q_gpu = bufs.team_probs[b, h, :n].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(q_gpu, q, rtol=1e-5, atol=1e-7 * q.max())
        draws, t, C = oracle.draw_with(sampler, q, M, seed, b, h)
        g_draws = bufs.draw_ids[b, h].cpu().numpy()
        i, o = compare_draws(g_draws, draws, t, C)
        assert o == 0, f"unit ({b},{h}): {o} draws differ outside the boundary window"
        inside, total = inside + i, total + M
        sel, rc = oracle.select_ex(draws, q, sampler)
        cnt = int(bufs.sel_count[b, h])
        g_sel = bufs.sel_ids[b, h].cpu().numpy()
        g_rc = bufs.pi[b, h].cpu().numpy().astype(np.float64)
        assert (g_sel[cnt:] == -1).all() and (g_rc[cnt:] == 0).all()
        if np.array_equal(g_draws, draws):
            assert np.array_equal(g_sel[:cnt], sel)
            np.testing.assert_allclose(g_rc[:cnt], rc, rtol=TOL_PI)
        units.append(((b, h), sel, rc))
        sel_t[b, h] = -1
        sel_t[b, h, :sel.size] = torch.from_numpy(sel).cuda()
        cnt_t[b, h] = sel.size
        rc_t[b, h] = 0.0
        rc_t[b, h, :sel.size] = torch.from_numpy(rc.astype(np.float32)).cuda()
    assert inside <= BOUNDARY_SHARE * total
    ab = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, sel_t,
                            cnt_t, rc_t)
    torch.cuda.synchronize()
    assert ab.status() == 0
    G, tol = cfg.group, TOL_OUT[cfg.dtype]
    fused = 0
    for (b, h), sel, rc in units:
        want = oracle.attend(pr, b, h, sel, rc)
        got = ab.out[b, h * G:(h + 1) * G].cpu().numpy()
        assert np.abs(got - want).max() <= tol, (b, h)
        if int(db.sel_count[b, h]) == sel.size and np.array_equal(
                db.sel_ids[b, h, :sel.size].cpu().numpy(), sel):
            got = db.out[b, h * G:(h + 1) * G].cpu().numpy()
            assert np.abs(got - want).max() <= tol, (b, h)
            fused += 1
    assert fused >= 1
