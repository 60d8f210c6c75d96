"""The steps on either side of the decode path: tokens appended one at a time
(santa_append_kv) between decode steps.

- The appended K/V rows land in the right paged slots.
- The representatives stay bit-identical to santa_build_reps on the grown cache, and within
  the parity tolerance of the oracle's means.
- A decode loop (append, decode, repeat) keeps matching the oracle on identical sampled sets
  as the sequences grow across page boundaries.
- A sampled set held over later steps (one refresh, then attention only) matches the
  oracle's attention over the same held set on the grown cache.
"""
import numpy as np
import pytest
import torch

import oracle
import sampled_sparse_decode_gb300 as santa
from sampled_sparse_decode_gb300 import workloads as W
from helpers import TOL_OUT, DeviceWorkload, to_torch

pytestmark = pytest.mark.gpu


def _grown(name, lens, **kw):
    wl = W.generate(name, seq_lens=lens, invalid_fill=float("nan"), batch=len(lens), **kw)
    return wl, DeviceWorkload(wl)


def _new_tokens(wl, step):
    """Seeded new K/V rows [B][Hkv][d] in the workload's dtype (bf16 rounded to nearest even)."""
    cfg = wl.cfg
    rng = np.random.default_rng([77, step])
    k = rng.standard_normal((cfg.batch, cfg.kv_heads, cfg.head_dim)).astype(np.float32)
    v = rng.standard_normal((cfg.batch, cfg.kv_heads, cfg.head_dim)).astype(np.float32)
    if cfg.dtype == "bf16":
        return W.f32_to_bf16_bits(k), W.f32_to_bf16_bits(v)
    return k, v


def _page_fill(page_table, lens, T, P):
    fill = np.zeros(P, dtype=np.int32)
    for b, L in enumerate(lens):
        for i in range(-(-int(L) // T)):
            fill[page_table[b, i]] = min(T, int(L) - i * T)
    return fill


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("name,extra", [
    ("qwen7b_32k_b8_m64", {}),
    ("llama8b_paged_32k_b16_m32", dict(num_pages=80)),
    ("tiny_f32", dict(q_heads=4, kv_heads=2, team_size=64)),
])
def test_appended_tokens_and_representatives(name, extra):
    T = extra.get("team_size", 128)
    lens0 = [1000, 760, T - 8, 2000]
    wl, dw = _grown(name, lens0, **extra)
    cfg = wl.cfg
    P = wl.k_pool.shape[0]
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    lens = [dw.seq_lens.clone(), torch.empty_like(dw.seq_lens)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    steps = 40
    written = []
    for s in range(steps):
        k_new, v_new = _new_tokens(wl, s)
        santa.santa_append_kv(to_torch(k_new), to_torch(v_new), dw.k_pool, dw.v_pool, reps,
                              dw.page_table, lens[s % 2], lens[(s + 1) % 2], status)
        written.append((k_new, v_new))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    final = lens[steps % 2].cpu().numpy()
    assert (final == np.array(lens0) + steps).all()
    # the rows are where they belong
    k_pool, v_pool = _host(dw.k_pool), _host(dw.v_pool)
    for s, (k_new, v_new) in enumerate(written):
        for b, L in enumerate(lens0):
            pos = L + s
            page = wl.page_table[b, pos // T]
            assert np.array_equal(k_pool[page, :, pos % T], k_new[b])
            assert np.array_equal(v_pool[page, :, pos % T], v_new[b])
    # representatives: bit-identical to a full rebuild, and within tolerance of the oracle
    fill = _page_fill(wl.page_table, final, T, P)
    rebuilt = santa.santa_build_reps(dw.k_pool, torch.from_numpy(fill).cuda())
    torch.cuda.synchronize()
    assert torch.equal(rebuilt, reps)
    pr = oracle.Problem(wl.q, k_pool, v_pool, wl.page_table, final)
    want = oracle.build_reps(pr, fill)
    np.testing.assert_allclose(reps.cpu().numpy().astype(np.float64), want, rtol=1e-5,
                               atol=1e-6 * np.abs(want).max())


def test_decode_loop_matches_oracle_as_sequences_grow():
    lens0 = [1000, 250, 127]
    wl, dw = _grown("qwen7b_32k_b8_m64", lens0, seq_len=1536)
    cfg = wl.cfg
    M = cfg.draws
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    lens = [dw.seq_lens.clone(), torch.empty_like(dw.seq_lens)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rng = np.random.default_rng(5)
    for s in range(24):
        k_new, v_new = _new_tokens(wl, 1000 + s)
        santa.santa_append_kv(to_torch(k_new), to_torch(v_new), dw.k_pool, dw.v_pool, reps,
                              dw.page_table, lens[s % 2], lens[(s + 1) % 2], status)
        cur = lens[(s + 1) % 2]
        q = W.f32_to_bf16_bits(q_rng.standard_normal(wl.q.shape).astype(np.float32))
        qd = to_torch(q)
        bufs = santa.santa_decode(qd, dw.k_pool, dw.v_pool, reps, dw.page_table, cur, M, s)
        if s in (0, 5, 23):
            torch.cuda.synchronize()
            assert bufs.status() == 0 and int(status.item()) == 0
            L = cur.cpu().numpy()
            pr = oracle.Problem(q, _host(dw.k_pool), _host(dw.v_pool), wl.page_table, L)
            fill = _page_fill(wl.page_table, L, cfg.team_size, wl.k_pool.shape[0])
            reps_o = oracle.build_reps(pr, fill)
            for b in range(cfg.batch):
                for h in range(cfg.kv_heads):
                    r = oracle.decode(pr, reps_o, M, s, b, h)
                    cnt = int(bufs.sel_count[b, h])
                    if cnt == r.sel.size and np.array_equal(
                            bufs.sel_ids[b, h, :cnt].cpu().numpy(), r.sel):
                        G = cfg.group
                        got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
                        assert np.abs(got - r.out).max() <= TOL_OUT["bf16"]
    torch.cuda.synchronize()
    assert (lens[24 % 2].cpu().numpy() == np.array(lens0) + 24).all()


def test_held_set_across_appends_matches_oracle():
    """A sampled set held over later steps (sampled once, then santa_attend with each step's
    own query on the grown cache): the outputs match the oracle's attention over the same
    held set and inclusion probabilities.  Sequences 1 and 2 open a new team during the
    hold, which the held set does not contain."""
    lens0 = [1000, 250, 127]
    wl, dw = _grown("qwen7b_32k_b8_m64", lens0, seq_len=1536)
    cfg = wl.cfg
    M, G = cfg.draws, cfg.group
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    held = santa.santa_sample(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                              M, 3)
    lens = [dw.seq_lens.clone(), torch.empty_like(dw.seq_lens)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rng = np.random.default_rng(6)
    checked = 0
    for s in range(24):
        k_new, v_new = _new_tokens(wl, 2000 + s)
        santa.santa_append_kv(to_torch(k_new), to_torch(v_new), dw.k_pool, dw.v_pool, reps,
                              dw.page_table, lens[s % 2], lens[(s + 1) % 2], status)
        cur = lens[(s + 1) % 2]
        q = W.f32_to_bf16_bits(q_rng.standard_normal(wl.q.shape).astype(np.float32))
        bufs = santa.santa_attend(to_torch(q), dw.k_pool, dw.v_pool, dw.page_table, cur,
                                  held.sel_ids, held.sel_count, held.pi)
        if s in (4, 23):
            torch.cuda.synchronize()
            assert bufs.status() == 0 and held.status() == 0 and int(status.item()) == 0
            L = cur.cpu().numpy()
            pr = oracle.Problem(q, _host(dw.k_pool), _host(dw.v_pool), wl.page_table, L)
            for b in range(cfg.batch):
                for h in range(cfg.kv_heads):
                    cnt = int(held.sel_count[b, h])
                    sel = held.sel_ids[b, h, :cnt].cpu().numpy()
                    pi = held.pi[b, h, :cnt].cpu().numpy().astype(np.float64)
                    assert sel.max() < -(-lens0[b] // cfg.team_size)
                    want = oracle.attend(pr, b, h, sel, pi)
                    got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
                    assert np.abs(got - want).max() <= TOL_OUT["bf16"]
                    checked += 1
    assert checked == 2 * cfg.batch * cfg.kv_heads
    final = lens[24 % 2].cpu().numpy()
    T = cfg.team_size
    assert -(-final[1] // T) > -(-lens0[1] // T) and -(-final[2] // T) > -(-lens0[2] // T)


def test_append_reports_full_sequences_and_bad_pages():
    wl, dw = _grown("tiny_f32", [64 * 32, 100])          # sequence 0 fills its last page
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k_new, v_new = _new_tokens(wl, 0)
    nxt = torch.empty_like(dw.seq_lens)
    santa.santa_append_kv(to_torch(k_new), to_torch(v_new), dw.k_pool, dw.v_pool, reps,
                          dw.page_table, dw.seq_lens, nxt, status)
    torch.cuda.synchronize()
    assert int(status.item()) & santa.DEV_BAD_SEQLEN
    assert int(nxt[1]) == 101
    pt = dw.page_table.clone()
    pt[1, 100 // 64] = -5
    status.zero_()
    santa.santa_append_kv(to_torch(k_new), to_torch(v_new), dw.k_pool, dw.v_pool, reps, pt,
                          dw.seq_lens, nxt, status)
    torch.cuda.synchronize()
    assert int(status.item()) & santa.DEV_BAD_PAGE
