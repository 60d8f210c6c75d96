"""GPU parity of value-row sampling inside the sampled teams (santa_attend_vs) against the
oracle, on the oracle's sampled teams and weights.

Drawn rows bit-exact except draws whose oracle point lies within the CDF-boundary window
(counted, < 1e-4 of draws); outputs of units whose rows all match within 1e-5 (fp32) /
2e-3 (bf16) max-abs of the oracle's value-sampled estimate.
"""
import numpy as np
import pytest
import torch

import oracle
import sampled_sparse_decode_gb300 as santa
from helpers import BOUNDARY_SHARE, TOL_OUT, DeviceWorkload, compare_draws, problem
from test_gpu_parity import SMALL, make

pytestmark = pytest.mark.gpu


def _oracle_sets(wl, pr, reps_o, M, seed):
    cfg = wl.cfg
    sel_t = torch.full((cfg.batch, cfg.kv_heads, M), -1, dtype=torch.int32)
    cnt_t = torch.zeros((cfg.batch, cfg.kv_heads), dtype=torch.int32)
    pi_t = torch.zeros((cfg.batch, cfg.kv_heads, M), dtype=torch.float32)
    sets = {}
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            p = oracle.team_probs(pr, reps_o, b, h)
            d, _, _ = oracle.draw(p, M, seed, b, h)
            s, pi = oracle.select(d, p)
            sel_t[b, h, :s.size] = torch.from_numpy(s)
            cnt_t[b, h] = s.size
            pi_t[b, h, :s.size] = torch.from_numpy(pi.astype(np.float32))
            sets[(b, h)] = (s, pi.astype(np.float32).astype(np.float64))
    return sel_t.cuda(), cnt_t.cuda(), pi_t.cuda(), sets


@pytest.mark.parametrize("name", ["tiny_f32", "qwen_b2_ragged", "llama_paged_b4",
                                  "bf16_d64_t64", "f32_d128_g8"])
@pytest.mark.parametrize("S", [8, 48])
def test_value_sampled_attention_parity(name, S):
    wl = make(SMALL[name])
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr, wl.page_fill)
    M, seed = cfg.draws, 2718
    sel_t, cnt_t, pi_t, sets = _oracle_sets(wl, pr, reps_o, M, seed)
    bufs, vids = santa.santa_attend_vs(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens,
                                       sel_t, cnt_t, pi_t, S, seed + 1, value_ids=True)
    torch.cuda.synchronize()
    assert bufs.status() == 0
    vids = vids.cpu().numpy()
    G, tol = cfg.group, TOL_OUT[cfg.dtype]
    inside = total = compared = 0
    for (b, h), (s, pi) in sets.items():
        all_match = True
        for c, team in enumerate(s):
            idx, t, C = oracle.vs_draw(pr, b, h, int(team), S, seed + 1)
            i, o = compare_draws(vids[b, h, c], idx, t, C)
            assert o == 0, f"unit ({b},{h}) team {team}: {o} row draws outside the window"
            inside, total = inside + i, total + S
            all_match &= bool(np.array_equal(vids[b, h, c], idx))
        if all_match:
            want, idx_o = oracle.attend_vs(pr, b, h, s, pi, S, seed + 1)
            assert np.array_equal(idx_o, vids[b, h, :s.size])
            got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
            assert np.abs(got - want).max() <= tol, (b, h, np.abs(got - want).max())
            compared += 1
    assert inside <= BOUNDARY_SHARE * total
    assert compared >= 0.9 * len(sets)


def test_value_sampling_arguments_and_bad_sets():
    wl = make(SMALL["tiny_f32"])
    dw = DeviceWorkload(wl)
    sel = torch.tensor([[[0, 3, 5, -1, -1, -1, -1, -1]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[3]], dtype=torch.int32, device="cuda")
    pi = torch.tensor([[[0.5, 0.7, 1.0, 0, 0, 0, 0, 0]]], dtype=torch.float32, device="cuda")
    for S in (0, 257):
        with pytest.raises(santa.SantaError, match="unsupported"):
            santa.santa_attend_vs(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, sel,
                                  cnt, pi, S, 1)
    bufs, _ = santa.santa_attend_vs(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens,
                                    sel, cnt, pi, 16, 1)
    torch.cuda.synchronize()
    assert bufs.status() == 0 and torch.isfinite(bufs.out).all()
    bad = sel.clone()
    bad[0, 0, 1] = 99
    bufs, _ = santa.santa_attend_vs(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens,
                                    bad, cnt, pi, 16, 1)
    torch.cuda.synchronize()
    assert bufs.status() & santa.DEV_BAD_SEL
    assert torch.isfinite(bufs.out).all()


@pytest.mark.parametrize("name", ["qwen7b_32k_b1_m31", "llama8b_paged_32k_b16_m32"])
def test_value_sampling_at_full_size(name):
    """Value-row sampling on a full-size workload, every unit's sampled set from the GPU's
    own sampling launch but the oracle's sets and weights on 8 units spread over the batch
    and the heads: drawn rows by the window rule, outputs where every row matches."""
    from helpers import full_oracle_reps, full_workload
    from test_gpu_parity import spread_units
    wl = full_workload(name)
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = full_oracle_reps(name)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    M, seed, S = cfg.draws, 515, 16
    sb = santa.santa_sample(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                            seed)
    torch.cuda.synchronize()
    sel_t, cnt_t, pi_t = sb.sel_ids.clone(), sb.sel_count.clone(), sb.pi.clone()
    sets = {}
    for b, h in spread_units(cfg.batch, cfg.kv_heads):
        p = oracle.team_probs(pr, reps_o, b, h)
        d, _, _ = oracle.draw(p, M, seed, b, h)
        s, pi = oracle.select(d, p)
        sel_t[b, h] = -1
        sel_t[b, h, :s.size] = torch.from_numpy(s).cuda()
        cnt_t[b, h] = s.size
        pi_t[b, h] = 0.0
        pi_t[b, h, :s.size] = torch.from_numpy(pi.astype(np.float32)).cuda()
        sets[(b, h)] = (s, pi.astype(np.float32).astype(np.float64))
    bufs, vids = santa.santa_attend_vs(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens,
                                       sel_t, cnt_t, pi_t, S, seed + 1, value_ids=True)
    torch.cuda.synchronize()
    assert bufs.status() == 0 and torch.isfinite(bufs.out).all()
    vids = vids.cpu().numpy()
    G, tol = cfg.group, TOL_OUT[cfg.dtype]
    inside = total = compared = 0
    for (b, h), (s, pi) in sets.items():
        all_match = True
        for c, team in enumerate(s):
            idx, t, C = oracle.vs_draw(pr, b, h, int(team), S, seed + 1)
            i, o = compare_draws(vids[b, h, c], idx, t, C)
            assert o == 0, f"unit ({b},{h}) team {team}: {o} row draws outside the window"
            inside, total = inside + i, total + S
            all_match &= bool(np.array_equal(vids[b, h, c], idx))
        if all_match:
            want, _ = oracle.attend_vs(pr, b, h, s, pi, S, seed + 1)
            got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
            assert np.abs(got - want).max() <= tol, (b, h, np.abs(got - want).max())
            compared += 1
    assert inside <= BOUNDARY_SHARE * total
    assert compared >= 0.75 * len(sets)
