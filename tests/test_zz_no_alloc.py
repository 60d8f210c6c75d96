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
])
def test_noalloc_matches_decode_on_two_calls(name, overrides):
    wl = W.generate(name, **overrides)
    cfg = wl.cfg
    dw = DeviceWorkload(wl)
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
    cap = santa.santa_noalloc_scratch_bytes()
    need = santa.santa_decode_workspace_min_bytes(512, 2, 1, 64, 64, 16384, 4096)
    assert need > cap
    wl = W.generate("tiny_f32")
    dw = DeviceWorkload(wl)
    reps = santa.santa_build_reps(dw.k_pool)
    B = 512
    q = dw.q.expand(B, -1, -1).contiguous()
    pt = dw.page_table.expand(B, -1).contiguous()
    pt = torch.nn.functional.pad(pt, (0, 16384 - pt.shape[1]))
    lens = dw.seq_lens.expand(B).contiguous()
    bufs = DecodeBuffers.allocate(q.dtype, B, 2, 1, 64, 64, 16384, 4096)
    with pytest.raises(santa.SantaError, match="scratch"):
        santa.santa_decode_noalloc(q, dw.k_pool, dw.v_pool, reps, pt, lens, 4096, 1, bufs)
