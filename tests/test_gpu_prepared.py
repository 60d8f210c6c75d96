"""The binding's fast path for decode loops: PreparedDecode (arguments marshalled once),
packed DecodeBuffers with a host mirror, and StepInputs.  The kernel and its arguments are
the same as santa_decode's, so the results must be bit-identical to santa_decode's."""
import numpy as np
import pytest
import torch

import sampled_sparse_decode_gb300 as santa
from sampled_sparse_decode_gb300 import workloads as W
from helpers import DeviceWorkload

pytestmark = pytest.mark.gpu


def _same(a, b):
    for f in ("out", "draw_ids", "sel_ids", "sel_count", "pi"):
        x, y = getattr(a, f), getattr(b, f)
        if f in ("sel_ids", "pi"):       # only the first sel_count slots are defined
            cnt = a.sel_count
            m = torch.arange(x.shape[-1], device=x.device) < cnt[..., None]
            x, y = x[m], y[m]
        assert torch.equal(x, y), f


def test_prepared_packed_matches_santa_decode():
    wl = W.generate("qwen7b_32k_b8_m64", batch=3, seq_len=5000)
    dw = DeviceWorkload(wl)
    cfg = wl.cfg
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    inp = santa.StepInputs.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.head_dim,
                                    wl.max_teams)
    inp.host_q.copy_(dw.q.cpu())
    inp.host_page_table.copy_(dw.page_table.cpu())
    inp.host_seq_lens.copy_(dw.seq_lens.cpu())
    inp.upload()
    pbufs = santa.DecodeBuffers.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.kv_heads,
                                         cfg.head_dim, cfg.team_size, wl.max_teams, cfg.draws,
                                         packed=True)
    prep = santa.santa_decode_prepared(inp.q, dw.k_pool, dw.v_pool, reps, inp.page_table,
                                       inp.seq_lens, cfg.draws, bufs=pbufs)
    host = pbufs.host_mirror()
    for seed in (0, 7, 123456789012345):
        prep.run(seed)
        pbufs.download(host)
        ref = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                                 cfg.draws, seed)
        torch.cuda.synchronize()
        assert pbufs.status() == 0 and ref.status() == 0
        _same(pbufs, ref)
        for f in ("out", "draw_ids", "sel_ids", "sel_count", "pi"):
            assert torch.equal(getattr(host, f), getattr(pbufs, f).cpu()), f
    # new query contents through the same storage
    q2 = W.f32_to_bf16_bits(np.random.default_rng(3).standard_normal(wl.q.shape)
                            .astype(np.float32))
    inp.host_q.copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16))
    inp.upload()
    prep.run(11)
    ref = santa.santa_decode(inp.q.clone(), dw.k_pool, dw.v_pool, reps, dw.page_table,
                             dw.seq_lens, cfg.draws, 11)
    torch.cuda.synchronize()
    _same(pbufs, ref)


def test_host_step_matches_santa_decode():
    """santa_decode_host through PreparedDecode.run_host: one upload, the decode, one
    download of outputs and status, and the wait, all in one call."""
    wl = W.generate("llama8b_paged_32k_b16_m32", batch=2, seq_len=3000, num_pages=64)
    dw = DeviceWorkload(wl)
    cfg = wl.cfg
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    inp = santa.StepInputs.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.head_dim,
                                    wl.max_teams)
    inp.host_q.copy_(dw.q.cpu())
    inp.host_page_table.copy_(dw.page_table.cpu())
    inp.host_seq_lens.copy_(dw.seq_lens.cpu())
    pbufs = santa.DecodeBuffers.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.kv_heads,
                                         cfg.head_dim, cfg.team_size, wl.max_teams, cfg.draws,
                                         packed=True)
    host = pbufs.host_mirror()
    prep = santa.santa_decode_prepared(inp.q, dw.k_pool, dw.v_pool, reps, inp.page_table,
                                       inp.seq_lens, cfg.draws, bufs=pbufs)
    for seed in (1, 2):
        prep.run_host(seed, inp, host)
        assert int(host.device_status[0]) == 0
        ref = santa.santa_decode(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table, dw.seq_lens,
                                 cfg.draws, seed)
        torch.cuda.synchronize()
        for f in ("out", "draw_ids", "sel_count"):
            assert torch.equal(getattr(host, f), getattr(ref, f).cpu()), f
        cnt = host.sel_count
        m = torch.arange(cfg.draws) < cnt[..., None]
        assert torch.equal(host.sel_ids[m], ref.sel_ids.cpu()[m])
        assert torch.equal(host.pi[m], ref.pi.cpu()[m])
    # a bad page id reaches the host through the packed status word
    inp.host_page_table[1, 0] = dw.k_pool.shape[0] + 5
    prep.run_host(3, inp, host)
    assert int(host.device_status[0]) & santa.DEV_BAD_PAGE
    with pytest.raises(santa.SantaError):
        santa.santa_decode_prepared(dw.q, dw.k_pool, dw.v_pool, reps, dw.page_table,
                                    dw.seq_lens, cfg.draws, bufs=pbufs).run_host(1, inp, host)


def test_host_step_copy_routes_agree():
    """santa_decode_host moves the slabs with its own copy kernels when the host buffers are
    page-locked, mapped and 16-byte aligned, and with the copy engine otherwise (pageable
    memory, unaligned pointers).  Every route gives the same host bytes, and new host
    contents written between calls are the ones the step reads."""
    import ctypes
    from sampled_sparse_decode_gb300 import binding as Bn
    wl = W.generate("qwen7b_32k_b8_m64", batch=2, seq_len=4000)
    dw = DeviceWorkload(wl)
    cfg = wl.cfg
    reps = santa.santa_build_reps(dw.k_pool, dw.page_fill)
    inp = santa.StepInputs.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.head_dim,
                                    wl.max_teams)
    inp.host_page_table.copy_(dw.page_table.cpu())
    inp.host_seq_lens.copy_(dw.seq_lens.cpu())
    pbufs = santa.DecodeBuffers.allocate(dw.q.dtype, cfg.batch, cfg.q_heads, cfg.kv_heads,
                                         cfg.head_dim, cfg.team_size, wl.max_teams, cfg.draws,
                                         packed=True)
    prep = santa.santa_decode_prepared(inp.q, dw.k_pool, dw.v_pool, reps, inp.page_table,
                                       inp.seq_lens, cfg.draws, bufs=pbufs)
    n_in, n_out = inp.slab.numel(), pbufs.outputs.numel()
    stream = torch.cuda.current_stream()

    def step(seed, host_in, host_out):
        prep._a.seed = seed
        rc = Bn.lib().santa_decode_host(ctypes.byref(prep._a), host_in.data_ptr(),
                                        inp.slab.data_ptr(), n_in, host_out.data_ptr(),
                                        pbufs.outputs.data_ptr(), n_out, stream.cuda_stream)
        assert rc == 0
        return host_out.clone()

    pinned_in = torch.empty(n_in + 16, dtype=torch.uint8, pin_memory=True)
    pinned_out = torch.empty(n_out + 16, dtype=torch.uint8, pin_memory=True)
    pageable_in = torch.empty(n_in, dtype=torch.uint8)
    pageable_out = torch.empty(n_out, dtype=torch.uint8)
    assert pinned_in.data_ptr() % 16 == 0 and pinned_out.data_ptr() % 16 == 0
    route = Bn.lib().santa_host_copy_route
    assert route(pinned_in.data_ptr(), inp.slab.data_ptr(), n_in) == 1
    assert route(pinned_out.data_ptr(), pbufs.outputs.data_ptr(), n_out) == 1
    assert route(inp.host_slab.data_ptr(), inp.slab.data_ptr(), n_in) == 1
    assert route(pageable_in.data_ptr(), inp.slab.data_ptr(), n_in) == 0
    assert route(pinned_in.data_ptr() + 8, inp.slab.data_ptr(), n_in) == 0
    # a range that runs past its pinned allocation takes the copy engine (nothing is copied
    # by this query)
    assert route(pinned_in.data_ptr(), inp.slab.data_ptr(),
                 (pinned_in.untyped_storage().nbytes() + (1 << 20)) // 16 * 16) == 0
    rng = np.random.default_rng(11)
    for trial in range(3):
        # new query contents for every trial, through the same host storage
        q = W.f32_to_bf16_bits(rng.standard_normal(wl.q.shape).astype(np.float32))
        inp.host_q.copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16))
        src = inp.host_slab
        routes = {
            "mapped": (pinned_in[:n_in], pinned_out[:n_out]),
            "pageable": (pageable_in, pageable_out),
            "unaligned": (pinned_in[8:8 + n_in], pinned_out[8:8 + n_out]),
        }
        got = {}
        for name, (hin, hout) in routes.items():
            hin.copy_(src)
            hout.fill_(0xA5)
            got[name] = step(40 + trial, hin, hout)
        ref = santa.santa_decode(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16)
                                 .to(dw.q.device), dw.k_pool, dw.v_pool, reps, dw.page_table,
                                 dw.seq_lens, cfg.draws, 40 + trial)
        torch.cuda.synchronize()
        assert ref.status() == 0
        for name in ("pageable", "unaligned"):
            assert torch.equal(got[name], got["mapped"]), name
        host = pbufs.host_mirror()
        host.slab.copy_(got["mapped"])
        assert int(host.device_status[0]) == 0
        assert torch.equal(host.out, ref.out.cpu())
        assert torch.equal(host.draw_ids, ref.draw_ids.cpu())
        assert torch.equal(host.sel_count, ref.sel_count.cpu())
