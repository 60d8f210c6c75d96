"""Packed step buffers of the binding (CPU): DecodeBuffers(packed=True) carves the five
outputs and the device status word out of one slab, host_mirror() gives host buffers of the same layout, and
StepInputs does the same for a step's inputs, so one copy moves each side.  Checked here:
shapes and dtypes, 16-byte alignment of every view, no overlap, and that a copy of the slab
moves every view's contents."""
import pytest
import torch

from sampled_sparse_decode_gb300 import binding as Bn


def _views_ok(slab, views):
    base = slab.data_ptr()
    spans = []
    for v in views:
        off = v.data_ptr() - base
        assert off % 16 == 0
        end = off + v.numel() * v.element_size()
        assert 0 <= off and end <= slab.numel()
        spans.append((off, end))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))


def _packed(B, Hq, Hkv, d, M, packed=True):
    """The outputs as DecodeBuffers.allocate lays them out (the workspace size query needs a
    GPU, so the scratch fields are stand-ins here)."""
    v, slab = Bn._output_views(B, Hq, Hkv, d, M, "cpu", packed)
    return Bn.DecodeBuffers(out=v[0], draw_ids=v[1], sel_ids=v[2], sel_count=v[3], pi=v[4],
                            team_probs=None, workspace=torch.zeros(16, dtype=torch.uint8),
                            device_status=v[5], outputs=slab)


@pytest.mark.parametrize("B,Hq,Hkv,d,M", [(3, 28, 4, 128, 31), (1, 2, 1, 64, 7)])
def test_packed_outputs_layout_and_round_trip(B, Hq, Hkv, d, M):
    bufs = _packed(B, Hq, Hkv, d, M)
    outs = [bufs.out, bufs.draw_ids, bufs.sel_ids, bufs.sel_count, bufs.pi]
    assert [tuple(x.shape) for x in outs] == [(B, Hq, d), (B, Hkv, M), (B, Hkv, M), (B, Hkv),
                                              (B, Hkv, M)]
    assert [x.dtype for x in outs] == [torch.float32, torch.int32, torch.int32, torch.int32,
                                       torch.float32]
    _views_ok(bufs.outputs, outs + [bufs.device_status])
    assert bufs.device_status.shape == (1,) and int(bufs.device_status[0]) == 0
    g = torch.Generator().manual_seed(1)
    bufs.out.copy_(torch.randn(bufs.out.shape, generator=g))
    bufs.draw_ids.copy_(torch.randint(0, 99, bufs.draw_ids.shape, generator=g))
    bufs.sel_ids.copy_(torch.randint(0, 99, bufs.sel_ids.shape, generator=g))
    bufs.sel_count.copy_(torch.randint(0, 99, bufs.sel_count.shape, generator=g))
    bufs.pi.copy_(torch.rand(bufs.pi.shape, generator=g))
    bufs.device_status.fill_(5)
    host = bufs.host_mirror()
    _views_ok(host.slab, [host.out, host.draw_ids, host.sel_ids, host.sel_count, host.pi,
                          host.device_status])
    bufs.download(host)
    for a, b in zip(outs, [host.out, host.draw_ids, host.sel_ids, host.sel_count, host.pi]):
        assert torch.equal(a, b)
    assert int(host.device_status[0]) == 5


def test_unpacked_buffers_have_no_mirror():
    bufs = _packed(1, 2, 1, 64, 4, packed=False)
    assert bufs.outputs is None
    with pytest.raises(Bn.SantaError):
        bufs.host_mirror()


def test_step_inputs_layout_and_upload():
    inp = Bn.StepInputs.allocate(torch.bfloat16, 2, 28, 128, 257, device="cpu")
    _views_ok(inp.slab, [inp.q, inp.page_table, inp.seq_lens])
    _views_ok(inp.host_slab, [inp.host_q, inp.host_page_table, inp.host_seq_lens])
    assert inp.q.shape == (2, 28, 128) and inp.q.dtype == torch.bfloat16
    assert inp.page_table.shape == (2, 257) and inp.seq_lens.shape == (2,)
    inp.host_q.copy_(torch.randn(2, 28, 128).to(torch.bfloat16))
    inp.host_page_table.copy_(torch.arange(514, dtype=torch.int32).view(2, 257))
    inp.host_seq_lens.copy_(torch.tensor([32768, 5], dtype=torch.int32))
    inp.upload()
    assert torch.equal(inp.q, inp.host_q)
    assert torch.equal(inp.page_table, inp.host_page_table)
    assert torch.equal(inp.seq_lens, inp.host_seq_lens)
