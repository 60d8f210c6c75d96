"""santa_decode_noalloc: santa_decode for callers that cannot allocate device memory (for
example a plug-in inside an engine that owns all GPU memory).  It runs the same decode with
the library's built-in scratch array; its outputs must match santa_decode's, on two calls in
a row (the array keeps the previous call's contents, which must not leak into the next).
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import sampled_sparse_decode_gb300 as santa
from sampled_sparse_decode_gb300 import workloads as W
from sampled_sparse_decode_gb300.binding import DecodeBuffers
from helpers import TOL_OUT, DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,overrides", [
    ("qwen7b_32k_b8_m64", dict(batch=3, seq_len=9000)),
    ("tiny_f32", {}),
    # 4096 draws over 4096 teams: the unit spans two clusters, whose partials go through
    # the scratch
    ("tiny_f32", dict(seq_len=4096 * 128, team_size=128, draws=4096)),
])
def test_noalloc_matches_decode_on_two_calls(name, overrides):
    wl = W.generate(name, **overrides)
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
    if cfg.draws == 4096:
        plan = santa.santa_decode_plan(dw.q, dw.k_pool, dw.page_table, cfg.draws, "decode",
                                       workspace_bytes=santa.santa_noalloc_scratch_bytes())
        assert plan["clusters_per_unit"] >= 2, plan
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    ref = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                             cfg.draws, 77)
    torch.cuda.synchronize()
    mt = dw.page_table.shape[1]
    bufs = DecodeBuffers.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.kv_heads,
                                  cfg.head_dim, cfg.team_size, mt, cfg.draws)
    bufs.workspace = torch.empty(0, dtype=torch.uint8, device="cuda")  # not used
    for _ in range(2):
        bufs.out.fill_(float("nan"))
        santa.santa_decode_noalloc(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table,
                                   dw.seq_lens, cfg.draws, 77, bufs)
        torch.cuda.synchronize()
        assert bufs.status() == 0
        assert torch.equal(bufs.sel_count, ref.sel_count)
        assert torch.equal(bufs.sel_ids, ref.sel_ids)
        assert torch.equal(bufs.draw_ids, ref.draw_ids)
        err = (bufs.out - ref.out).abs().max().item()
        assert err <= TOL_OUT[cfg.dtype], err


def test_noalloc_rejects_problems_beyond_its_scratch():
    """512 units of 4096 draws over 4096 teams need two clusters' partials per unit, more
    than the built-in scratch holds: the call is refused before anything runs."""
    B, Hq, Hkv, d, T, teams, M = 64, 64, 8, 128, 128, 4096, 4096
    cap = santa.santa_noalloc_scratch_bytes()
    assert santa.santa_decode_workspace_min_bytes(B, Hq, Hkv, d, T, teams, M) > cap
    dev = "cuda"
    q = torch.zeros((B, Hq, d), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((4, Hkv, T, d), dtype=torch.bfloat16, device=dev)
    reps = torch.zeros((4, Hkv, d), dtype=torch.float32, device=dev)
    pt = torch.zeros((B, teams), dtype=torch.int32, device=dev)
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    bufs = DecodeBuffers.allocate(q.dtype, B, Hq, Hkv, d, T, teams, M)
    with pytest.raises(santa.SantaError, match="scratch"):
        santa.santa_decode_noalloc(q, k, k, reps, pt, lens, M, 1, bufs)
