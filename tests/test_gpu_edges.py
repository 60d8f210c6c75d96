"""GPU edge cases: degenerate team distributions, extreme draw counts, workspace sizes,
device-side error reporting without faults, determinism, and the Philox cross-check
against CUDA's own curand_Philox4x32_10."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import sampled_sparse_decode_gb300 as santa
from sampled_sparse_decode_gb300 import workloads as W
from sampled_sparse_decode_gb300.binding import DecodeBuffers
from helpers import TOL_OUT, DeviceWorkload, problem

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def decode_vs_oracle(wl, M, seed, units=None, tol=None):
    """santa_decode vs the oracle's decode on every (or the given) unit; requires equal S."""
    dw = DeviceWorkload(wl)
    pr = problem(wl)
    reps_o = oracle.build_reps(pr, wl.page_fill)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    bufs = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens, M,
                              seed, team_probs=True)
    torch.cuda.synchronize()
    assert bufs.status() == 0
    tol = tol or TOL_OUT[wl.cfg.dtype]
    G = wl.cfg.group
    units = units or [(b, h) for b in range(wl.cfg.batch) for h in range(wl.cfg.kv_heads)]
    res = []
    for b, h in units:
        r = oracle.decode(pr, reps_o, M, seed, b, h)
        cnt = int(bufs.sel_count[b, h])
        assert cnt == r.sel.size and np.array_equal(bufs.sel_ids[b, h, :cnt].cpu().numpy(), r.sel)
        got = bufs.out[b, h * G:(h + 1) * G].cpu().numpy()
        assert np.abs(got - r.out).max() <= tol
        res.append(r)
    return bufs, res


def test_single_team_sequence():
    wl = W.generate("tiny_f32", seq_lens=[50], invalid_fill=float("nan"))
    bufs, (r,) = decode_vs_oracle(wl, 8, 3)
    assert int(bufs.sel_count[0, 0]) == 1 and float(bufs.pi[0, 0, 0]) == 1.0
    assert (bufs.draw_ids[0, 0] == 0).all()


def test_more_draws_than_teams_reaches_dense():
    """M = 4096 >> 32 teams with a near-uniform distribution: every team is sampled with
    pi = 1 and the estimate is dense attention."""
    wl = W.generate("tiny_f32")
    wl.q[:] = wl.q * np.float32(0.05)
    bufs, (r,) = decode_vs_oracle(wl, 4096, 5)
    assert int(bufs.sel_count[0, 0]) == 32
    assert (bufs.pi[0, 0, :32] == 1.0).all()
    dense = oracle.dense(problem(wl), 0, 0)
    assert np.abs(bufs.out[0].cpu().numpy() - dense).max() <= TOL_OUT["f32"]


def test_equal_scores_uniform_distribution():
    wl = W.generate("qwen7b_32k_b1_m31", seq_len=3000)
    wl.q[:] = 0
    bufs, _ = decode_vs_oracle(wl, 31, 11)
    n = wl.cfg.n_teams
    tp = bufs.team_probs[0, 0, :n].cpu().numpy()
    np.testing.assert_allclose(tp, 1.0 / n, rtol=1e-6)


def test_peaked_distribution_with_underflow():
    """A query 40x larger makes one team dominate and most team probabilities underflow to
    zero in fp32; zero-probability teams are never drawn."""
    wl = W.generate("qwen7b_32k_b1_m31", seq_len=8000)
    q = W.bf16_bits_to_f32(wl.q) * 40.0
    wl.q[:] = W.f32_to_bf16_bits(q)
    bufs, res = decode_vs_oracle(wl, 31, 13)
    tp = bufs.team_probs.cpu().numpy()
    for h in range(wl.cfg.kv_heads):
        drawn = bufs.draw_ids[0, h].cpu().numpy()
        assert (tp[0, h][drawn] > 0).all()


def test_workspace_of_minimum_size():
    """The smallest workspace the library accepts gives the same sampled sets and the same
    output (to rounding) as the default one, also for a unit whose work spans several
    clusters (4096 draws over 4096 teams)."""
    for name, over in [("qwen7b_32k_b8_m64", dict(batch=2, seq_len=5000)),
                       ("tiny_f32", dict(seq_len=4096 * 128, team_size=128, draws=4096))]:
        wl = W.generate(name, **over)
        dw = DeviceWorkload(wl)
        reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
        cfg = wl.cfg
        full = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table,
                                  dw.seq_lens, cfg.draws, 3)
        mt = dw.page_table.shape[1]
        small = DecodeBuffers.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.kv_heads,
                                       cfg.head_dim, cfg.team_size, mt, cfg.draws)
        small.workspace = torch.zeros(santa.santa_decode_workspace_min_bytes(
            cfg.batch, cfg.q_heads, cfg.kv_heads, cfg.head_dim, cfg.team_size, mt, cfg.draws),
            dtype=torch.uint8, device="cuda")
        santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                           cfg.draws, 3, bufs=small)
        torch.cuda.synchronize()
        assert full.status() == 0 and small.status() == 0
        assert torch.equal(full.sel_ids, small.sel_ids)
        assert (full.out - small.out).abs().max().item() <= 1e-5


def test_maximum_team_count():
    """The largest supported cache per sequence: max_teams = 16384 teams of 64 tokens
    (1M tokens, bf16, d = 64).  The sampling takes the largest cluster, 16 CTAs of 1024
    teams each, the most one CTA scores.  S and the output match the oracle for M = 64 and
    for the largest M, 4096 (whose sampled teams also span several clusters)."""
    wl = W.generate("tiny_f32", seq_len=16384 * 64, dtype="bf16", draws=64)
    assert wl.max_teams == 16384
    dw = DeviceWorkload(wl)
    plan = santa.santa_decode_plan(dw.q, dw.k_pool, dw.page_table, 64, "decode")
    assert plan["cluster"] == 16 and plan["teams_per_cta"] == 1024, plan
    for M, seed in ((64, 5), (4096, 6)):
        bufs, res = decode_vs_oracle(wl, M, seed)
        assert res[0].sel.size == int(bufs.sel_count[0, 0]) > M // 2


def test_repeated_calls_are_deterministic():
    """The workspace counters reset themselves: back-to-back calls on the same buffers give
    bit-identical outputs."""
    wl = W.generate("llama8b_paged_32k_b16_m32", batch=3, seq_len=7000, num_pages=200)
    dw = DeviceWorkload(wl)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    cfg = wl.cfg
    bufs = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                              cfg.draws, 21)
    first = bufs.out.clone()
    for _ in range(3):
        santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                           cfg.draws, 21, bufs=bufs)
    torch.cuda.synchronize()
    assert torch.equal(first, bufs.out)
    dense = santa.santa_dense_decode(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens)
    o1 = dense.out.clone()
    santa.santa_dense_decode(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, bufs=dense)
    torch.cuda.synchronize()
    assert torch.equal(o1, dense.out)


def test_bad_page_and_seq_len_are_reported_not_trapped():
    wl = W.generate("qwen7b_32k_b8_m64", batch=3, seq_len=2000)
    dw = DeviceWorkload(wl)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    P = dw.k_pool.shape[0]
    pt = dw.page_table.clone()
    pt[1, 3] = P + 5                               # sequence 1: one page id out of range
    lens = dw.seq_lens.clone()
    lens[2] = 0                                    # sequence 2: empty
    bufs = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, pt, lens, 64, 1,
                              team_probs=True)
    torch.cuda.synchronize()
    st = bufs.status()
    assert st & santa.DEV_BAD_PAGE and st & santa.DEV_BAD_SEQLEN
    assert (bufs.sel_count[2] == 0).all() and (bufs.out[2] == 0).all()
    assert (bufs.draw_ids[2] == -1).all()
    assert (bufs.team_probs[1, :, 3] == 0).all()  # the bad team is never drawn
    assert torch.isfinite(bufs.out).all()
    # sequence 0 is untouched by the errors of the others
    ref = santa.santa_decode(dw.q[:1].contiguous(), dw.k_pool, dw.v_pool, reps,
                             dw.page_table[:1].contiguous(), dw.seq_lens[:1].contiguous(), 64, 1)
    torch.cuda.synchronize()
    assert torch.equal(ref.sel_ids[0], bufs.sel_ids[0])
    assert (ref.out[0] - bufs.out[0]).abs().max().item() <= 1e-5


def test_bad_sampled_set_is_reported():
    wl = W.generate("tiny_f32")
    dw = DeviceWorkload(wl)
    sel = torch.tensor([[[0, 99, -1, -1]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[2]], dtype=torch.int32, device="cuda")
    pi = torch.tensor([[[0.5, 0.5, 0.0, 0.0]]], dtype=torch.float32, device="cuda")
    bufs = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, sel, cnt,
                              pi)
    torch.cuda.synchronize()
    assert bufs.status() & santa.DEV_BAD_SEL
    assert torch.isfinite(bufs.out).all()
    # 1 / weight must be finite and positive (above 1 is fine: Hansen-Hurwitz weights)
    for bad in (float("inf"), float("nan"), 0.0, -0.5):
        sel = torch.tensor([[[0, 3, -1, -1]]], dtype=torch.int32, device="cuda")
        pi = torch.tensor([[[1.7, bad, 0.0, 0.0]]], dtype=torch.float32, device="cuda")
        bufs = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, sel,
                                  cnt, pi)
        torch.cuda.synchronize()
        assert bufs.status() & santa.DEV_BAD_SEL, bad
    pi = torch.tensor([[[1.7, 0.3, 0.0, 0.0]]], dtype=torch.float32, device="cuda")
    bufs = santa.santa_attend(dw.q, dw.k_pool, dw.v_pool, dw.page_table, dw.seq_lens, sel, cnt, pi)
    torch.cuda.synchronize()
    assert bufs.status() == 0


def test_update_reps_matches_build():
    wl = W.generate("llama8b_paged_32k_b16_m32", batch=2, seq_len=3000, num_pages=100)
    dw = DeviceWorkload(wl)
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    # grow the last page of sequence 0 by one token and refresh just that page
    last = int(wl.page_table[0, -1])
    fill = dw.page_fill.clone()
    fill[last] += 1
    dw.k_pool[last, :, int(wl.page_fill[last])] = 1.5
    santa.santa_update_reps(dw.k_pool, torch.tensor([last], dtype=torch.int32, device="cuda"),
                            reps, fill)
    fresh = santa.santa_build_reps(dw.k_pool, fill)
    torch.cuda.synchronize()
    assert torch.equal(reps, fresh)


def test_device_philox_matches_curand():
    """The library's device Philox4x32-10 equals CUDA's curand_Philox4x32_10 bit for bit."""
    so = os.path.join(ROOT, "tests", "cuda", "philox_check.so")
    src = os.path.join(ROOT, "tests", "cuda", "philox_check.cu")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                        "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                        f"-I{ROOT}/include", f"-I{ROOT}/sampled_sparse_decode_gb300/csrc",
                        "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    n = 4096
    rng = np.random.default_rng(0)
    ctr = torch.from_numpy(rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64)
                           .astype(np.uint32).view(np.int32)).cuda()
    key = torch.from_numpy(rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64)
                           .astype(np.uint32).view(np.int32)).cuda()
    ours = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    ref = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    assert lib.philox_pair(ctypes.c_void_p(ctr.data_ptr()), ctypes.c_void_p(key.data_ptr()),
                           ctypes.c_void_p(ours.data_ptr()), ctypes.c_void_p(ref.data_ptr()),
                           n) == 0
    assert torch.equal(ours, ref)
    # and the oracle's Philox agrees with both on a few of them
    c = ctr.cpu().numpy().view(np.uint32)
    k = key.cpu().numpy().view(np.uint32)
    o = ours.cpu().numpy().view(np.uint32)
    for i in range(0, n, 257):
        assert np.array_equal(oracle.philox4x32_10(c[i], k[i]), o[i])
