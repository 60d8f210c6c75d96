"""Thin ctypes binding of libsanta.so: argument marshalling only.

Every function takes torch CUDA tensors, checks their dtypes/shapes/layout, fills the C
structure declared in include/santa.h and calls the entry point of the same name on the
current torch stream.  All computation happens in the library's kernels; if the library
cannot be loaded, the first call raises (there is no CPU fallback).

Shapes (as in the C header): q [B][Hq][d]; k_pool, v_pool [P][Hkv][T][d] (float32 or
bfloat16); reps [P][Hkv][d] float32; page_table [B][max_teams] int32; seq_lens [B] int32.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))

DEV_BAD_PAGE, DEV_BAD_SEQLEN, DEV_BAD_SEL, DEV_TIMEOUT = 1, 2, 4, 8
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}


class SantaError(RuntimeError):
    pass


class _DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("reps", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("dtype", ctypes.c_int), ("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("team_size", ctypes.c_int),
        ("max_teams", ctypes.c_int), ("num_draws", ctypes.c_int),
        ("num_pages", ctypes.c_int64), ("seed", ctypes.c_uint64),
        ("out", ctypes.c_void_p), ("draw_ids", ctypes.c_void_p), ("sel_ids", ctypes.c_void_p),
        ("sel_count", ctypes.c_void_p), ("pi", ctypes.c_void_p), ("team_probs", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("device_status", ctypes.c_void_p),
        ("sampler", ctypes.c_int32), ("mix_alpha", ctypes.c_float),
    ]


# Samplers (santa_sampler): i.i.d. draws with Horvitz-Thompson weights (the method),
# systematic draws with Horvitz-Thompson weights, i.i.d. draws with Hansen-Hurwitz weights.
SAMPLERS = {"iid_ht": 0, "systematic": 1, "iid_hh": 2}


_lib = None


def lib():
    """Load libsanta.so (building it from source first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        A = ctypes.POINTER(_DecodeArgs)
        sigs = {
            "santa_abi_version": (i32, []),
            "santa_status_string": (ctypes.c_char_p, [i32]),
            "santa_build_reps": (i32, [vp, i32, i64, i32, i32, i32, vp, vp, vp, vp]),
            "santa_update_reps": (i32, [vp, i32, i64, i32, i32, i32, vp, i32, vp, vp, vp, vp]),
            "santa_decode_workspace_bytes": (sz, [i32] * 8),
            "santa_decode_workspace_min_bytes": (sz, [i32] * 7),
            "santa_dense_workspace_bytes": (sz, [i32] * 7),
            "santa_sample": (i32, [A, vp]),
            "santa_attend_vs": (i32, [A, i32, vp, vp]),
            "santa_attend_vs_workspace_bytes": (sz, [i32] * 5),
            "santa_append_kv": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, i64, vp, vp, vp, vp,
                                      vp, vp, vp, vp]),
            "santa_attend": (i32, [A, vp]),
            "santa_decode": (i32, [A, vp]),
            "santa_dense_decode": (i32, [A, vp]),
            "santa_decode_noalloc": (i32, [A, vp]),
            "santa_decode_host": (i32, [A, vp, vp, sz, vp, vp, sz, vp]),
            "santa_host_copy_route": (i32, [vp, vp, sz]),
            "santa_decode_plan": (i32, [A, i32, vp]),
            "santa_decode_path": (i32, [A]),
            "santa_noalloc_scratch_bytes": (sz, []),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def santa_abi_version() -> int:
    return lib().santa_abi_version()


def santa_status_string(status: int) -> str:
    return lib().santa_status_string(status).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise SantaError(f"{what}: {santa_status_string(rc)} (status {rc})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _req(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise SantaError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise SantaError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise SantaError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise SantaError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return _DTYPES[dtype]


def santa_decode_workspace_bytes(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size,
                                 max_teams, num_draws) -> int:
    """dtype: torch.float32 / torch.bfloat16 (or 0 / 1)."""
    return lib().santa_decode_workspace_bytes(_dtype_code(dtype), batch, num_q_heads,
                                              num_kv_heads, head_dim, team_size, max_teams,
                                              num_draws)


def santa_decode_workspace_min_bytes(batch, num_q_heads, num_kv_heads, head_dim, team_size,
                                     max_teams, num_draws) -> int:
    return lib().santa_decode_workspace_min_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                  team_size, max_teams, num_draws)


def santa_dense_workspace_bytes(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size,
                                max_teams) -> int:
    return lib().santa_dense_workspace_bytes(_dtype_code(dtype), batch, num_q_heads,
                                             num_kv_heads, head_dim, team_size, max_teams)


def santa_build_reps(k_pool: torch.Tensor, page_fill: torch.Tensor | None = None,
                     reps: torch.Tensor | None = None, device_status: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Mean key of every (page, KV head) -> reps [P][Hkv][d] float32."""
    _req(k_pool, "k_pool", ndim=4)
    P, Hkv, T, d = k_pool.shape
    if k_pool.dtype not in _DTYPES:
        raise SantaError("k_pool must be float32 or bfloat16")
    if reps is None:
        reps = torch.empty((P, Hkv, d), dtype=torch.float32, device=k_pool.device)
    _req(reps, "reps", torch.float32)
    if page_fill is not None:
        _req(page_fill, "page_fill", torch.int32)
    _check(lib().santa_build_reps(_ptr(k_pool), _DTYPES[k_pool.dtype], P, Hkv, T, d,
                                  _ptr(page_fill), _ptr(reps), _ptr(device_status),
                                  _stream(stream)), "santa_build_reps")
    return reps


def santa_update_reps(k_pool: torch.Tensor, pages: torch.Tensor, reps: torch.Tensor,
                      page_fill: torch.Tensor | None = None,
                      device_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Recompute the representatives of the listed pages in place."""
    _req(k_pool, "k_pool", ndim=4)
    _req(pages, "pages", torch.int32, 1)
    _req(reps, "reps", torch.float32)
    P, Hkv, T, d = k_pool.shape
    _check(lib().santa_update_reps(_ptr(k_pool), _DTYPES[k_pool.dtype], P, Hkv, T, d,
                                   _ptr(pages), pages.numel(), _ptr(page_fill), _ptr(reps),
                                   _ptr(device_status), _stream(stream)), "santa_update_reps")
    return reps


def _carve(slab: torch.Tensor, specs):
    """Views of a flat uint8 tensor: one per (shape, dtype) in specs, each starting on a
    16-byte boundary, in order."""
    views, off = [], 0
    for shape, dtype in specs:
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        views.append(slab[off:off + nbytes].view(dtype).view(shape))
        off += (nbytes + 15) // 16 * 16
    return views


def _packed_bytes(specs) -> int:
    total = 0
    for shape, dtype in specs:
        n = 1
        for x in shape:
            n *= x
        total += (n * torch.empty((), dtype=dtype).element_size() + 15) // 16 * 16
    return total


def _host_slab(nbytes: int) -> torch.Tensor:
    """Page-locked when a GPU is present (asynchronous copies), plain memory otherwise."""
    return torch.empty(nbytes, dtype=torch.uint8, pin_memory=torch.cuda.is_available())


def _output_specs(batch, num_q_heads, num_kv_heads, head_dim, num_draws):
    """out, draw_ids, sel_ids, sel_count, pi and the device status word."""
    B, Hkv, M = batch, num_kv_heads, max(num_draws, 1)
    return [((B, num_q_heads, head_dim), torch.float32), ((B, Hkv, M), torch.int32),
            ((B, Hkv, M), torch.int32), ((B, Hkv), torch.int32), ((B, Hkv, M), torch.float32),
            ((1,), torch.int32)]


def _output_views(batch, num_q_heads, num_kv_heads, head_dim, num_draws, device, packed):
    """(out, draw_ids, sel_ids, sel_count, pi, device_status) and their slab (None unless
    packed).  The status word starts at zero."""
    specs = _output_specs(batch, num_q_heads, num_kv_heads, head_dim, num_draws)
    if not packed:
        views = [torch.empty(shape, dtype=dt, device=device) for shape, dt in specs[:-1]]
        return views + [torch.zeros(1, dtype=torch.int32, device=device)], None
    slab = torch.zeros(_packed_bytes(specs), dtype=torch.uint8, device=device)
    return _carve(slab, specs), slab


@dataclass
class HostOutputs:
    """Host copies of a packed DecodeBuffers' outputs and status word (views of `slab`)."""
    out: torch.Tensor
    draw_ids: torch.Tensor
    sel_ids: torch.Tensor
    sel_count: torch.Tensor
    pi: torch.Tensor
    device_status: torch.Tensor
    slab: torch.Tensor


@dataclass
class DecodeBuffers:
    """Outputs and scratch of one decode step for a fixed shape (reusable across steps)."""
    out: torch.Tensor          # [B][Hq][d] float32
    draw_ids: torch.Tensor     # [B][Hkv][M] int32
    sel_ids: torch.Tensor      # [B][Hkv][M] int32
    sel_count: torch.Tensor    # [B][Hkv] int32
    pi: torch.Tensor           # [B][Hkv][M] float32
    team_probs: torch.Tensor | None   # [B][Hkv][max_teams] float32
    workspace: torch.Tensor    # uint8
    device_status: torch.Tensor  # [1] int32
    outputs: torch.Tensor | None = None   # packed: the five outputs above as one uint8 slab

    @staticmethod
    def allocate(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size, max_teams,
                 num_draws, device="cuda", team_probs=False, dense=False,
                 packed=False) -> "DecodeBuffers":
        """dtype of q/K/V (torch.float32 or torch.bfloat16); sizes as in santa.h.  With
        packed=True, out, draw_ids, sel_ids, sel_count, pi and device_status are views of one
        slab (`outputs`, each view 16-byte aligned), so one copy brings them all to the host
        (host_mirror / download)."""
        B, Hkv, M = batch, num_kv_heads, max(num_draws, 1)
        ws = (santa_dense_workspace_bytes(dtype, B, num_q_heads, Hkv, head_dim, team_size,
                                          max_teams)
              if dense else
              santa_decode_workspace_bytes(dtype, B, num_q_heads, Hkv, head_dim, team_size,
                                           max_teams, M))
        if ws == 0:
            raise SantaError("unsupported shape for the workspace query")
        views, slab = _output_views(B, num_q_heads, Hkv, head_dim, M, device, packed)
        return DecodeBuffers(
            out=views[0], draw_ids=views[1], sel_ids=views[2], sel_count=views[3], pi=views[4],
            team_probs=(torch.empty((B, Hkv, max_teams), dtype=torch.float32, device=device)
                        if team_probs else None),
            workspace=torch.zeros(ws, dtype=torch.uint8, device=device),
            device_status=views[5],
            outputs=slab,
        )

    def host_mirror(self) -> HostOutputs:
        """Host buffers with the packed layout of this DecodeBuffers (packed=True only)."""
        if self.outputs is None:
            raise SantaError("host_mirror needs DecodeBuffers.allocate(..., packed=True)")
        B, Hq, d = self.out.shape
        _, Hkv, M = self.pi.shape
        specs = _output_specs(B, Hq, Hkv, d, M)
        slab = _host_slab(self.outputs.numel())
        return HostOutputs(*_carve(slab, specs), slab=slab)

    def download(self, host: HostOutputs, stream=None) -> HostOutputs:
        """One asynchronous device->host copy of the outputs and status into `host` on `stream`
        (the current stream by default); synchronise before reading it."""
        if self.outputs is None or host.slab.numel() != self.outputs.numel():
            raise SantaError("download needs a packed DecodeBuffers and its host_mirror()")
        if stream is None:
            host.slab.copy_(self.outputs, non_blocking=True)
        else:
            with torch.cuda.stream(stream):
                host.slab.copy_(self.outputs, non_blocking=True)
        return host

    def status(self) -> int:
        """Synchronise with the device and return the device status word."""
        return int(self.device_status.item())


@dataclass
class StepInputs:
    """The per-step inputs q [B][Hq][d], page_table [B][max_teams] and seq_lens [B] as views
    of one device slab, with host buffers of the same layout (host_q, host_page_table,
    host_seq_lens), so that one copy uploads a step's inputs."""
    q: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    host_q: torch.Tensor
    host_page_table: torch.Tensor
    host_seq_lens: torch.Tensor
    slab: torch.Tensor
    host_slab: torch.Tensor

    @staticmethod
    def allocate(dtype, batch, num_q_heads, head_dim, max_teams, device="cuda") -> "StepInputs":
        specs = [((batch, num_q_heads, head_dim), dtype), ((batch, max_teams), torch.int32),
                 ((batch,), torch.int32)]
        nbytes = _packed_bytes(specs)
        slab = torch.empty(nbytes, dtype=torch.uint8, device=device)
        host = _host_slab(nbytes)
        return StepInputs(*_carve(slab, specs), *_carve(host, specs), slab=slab,
                          host_slab=host)

    def upload(self, stream=None) -> "StepInputs":
        """One asynchronous host->device copy of the three host buffers on `stream`."""
        if stream is None:
            self.slab.copy_(self.host_slab, non_blocking=True)
        else:
            with torch.cuda.stream(stream):
                self.slab.copy_(self.host_slab, non_blocking=True)
        return self


class PreparedDecode:
    """santa_decode with its arguments checked and marshalled once, for steps that reuse
    the same tensors (a decode loop over persistent buffers).  run(seed) changes only the
    seed; the tensors' contents may change between runs, their storage may not."""

    def __init__(self, q, k_pool, v_pool, reps, page_table, seq_lens, num_draws: int,
                 bufs: DecodeBuffers | None = None, sampler: str = "iid_ht",
                 mix_alpha: float = 0.0, team_probs: bool = False):
        self.bufs = _bufs_for(q, k_pool, page_table, num_draws, bufs, team_probs)
        self._keep = (q, k_pool, v_pool, reps, page_table, seq_lens)
        self._a = _args(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws, 0,
                        self.bufs, sampler, mix_alpha)
        self._fn = lib().santa_decode
        self._aref = ctypes.byref(self._a)
        self._host_call = None      # (inputs, host, santa_decode_host's buffer arguments)

    def run(self, seed: int, stream=None) -> DecodeBuffers:
        self._a.seed = seed & 0xFFFFFFFFFFFFFFFF
        _check(self._fn(self._aref, _stream(stream)), "santa_decode")
        return self.bufs

    def run_host(self, seed: int, inputs: StepInputs, host: HostOutputs,
                 stream=None) -> HostOutputs:
        """One step through santa_decode_host: inputs.host_slab -> inputs.slab, the decode,
        bufs.outputs -> host.slab, then a wait for the stream.  The PreparedDecode must have
        been made on inputs' device views and packed DecodeBuffers; host.device_status holds
        the step's status word (sticky: zero it in the device slab to clear it)."""
        c = self._host_call
        if c is None or c[0] is not inputs or c[1] is not host:
            b = self.bufs
            if (b.outputs is None or host.slab.numel() != b.outputs.numel() or
                    self._a.q != inputs.q.data_ptr() or
                    self._a.page_table != inputs.page_table.data_ptr() or
                    self._a.seq_lens != inputs.seq_lens.data_ptr()):
                raise SantaError("run_host needs packed DecodeBuffers, their host_mirror() "
                                 "and a PreparedDecode made on the StepInputs' device views")
            # checked once per (inputs, host) pair: their storage may not change afterwards
            c = self._host_call = (inputs, host, lib().santa_decode_host,
                                   (inputs.host_slab.data_ptr(), inputs.slab.data_ptr(),
                                    inputs.slab.numel(), host.slab.data_ptr(),
                                    b.outputs.data_ptr(), b.outputs.numel()))
        self._a.seed = seed & 0xFFFFFFFFFFFFFFFF
        _check(c[2](self._aref, *c[3], _stream(stream)), "santa_decode_host")
        return host


def santa_decode_prepared(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws: int,
                          bufs: DecodeBuffers | None = None, sampler: str = "iid_ht",
                          mix_alpha: float = 0.0, team_probs: bool = False) -> PreparedDecode:
    """A PreparedDecode: santa_decode's checks and argument structure done once."""
    return PreparedDecode(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws, bufs,
                          sampler, mix_alpha, team_probs)


def _args(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws, seed,
          bufs: DecodeBuffers, sampler: str = "iid_ht", mix_alpha: float = 0.0) -> _DecodeArgs:
    _req(q, "q", ndim=3)
    _req(k_pool, "k_pool", ndim=4)
    _req(v_pool, "v_pool", ndim=4)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    if q.dtype not in _DTYPES or k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise SantaError("q, k_pool and v_pool must share one dtype (float32 or bfloat16)")
    if k_pool.shape != v_pool.shape:
        raise SantaError("k_pool and v_pool must have the same shape")
    if reps is not None:
        _req(reps, "reps", torch.float32, 3)
    B, Hq, d = q.shape
    P, Hkv, T, d2 = k_pool.shape
    if d2 != d or page_table.shape[0] != B or seq_lens.shape[0] != B:
        raise SantaError("shape mismatch between q, k_pool, page_table and seq_lens")
    a = _DecodeArgs()
    a.q, a.k_pool, a.v_pool, a.reps = _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(reps)
    a.page_table, a.seq_lens = _ptr(page_table), _ptr(seq_lens)
    a.dtype, a.batch, a.num_q_heads, a.num_kv_heads = _DTYPES[q.dtype], B, Hq, Hkv
    a.head_dim, a.team_size, a.max_teams, a.num_draws = d, T, page_table.shape[1], num_draws
    a.num_pages, a.seed = P, seed & 0xFFFFFFFFFFFFFFFF
    a.out, a.draw_ids, a.sel_ids = _ptr(bufs.out), _ptr(bufs.draw_ids), _ptr(bufs.sel_ids)
    a.sel_count, a.pi, a.team_probs = _ptr(bufs.sel_count), _ptr(bufs.pi), _ptr(bufs.team_probs)
    a.workspace, a.workspace_bytes = _ptr(bufs.workspace), bufs.workspace.numel()
    if sampler not in SAMPLERS:
        raise SantaError(f"unknown sampler {sampler!r} (one of {sorted(SAMPLERS)})")
    a.sampler, a.mix_alpha = SAMPLERS[sampler], float(mix_alpha)
    a.device_status = _ptr(bufs.device_status)
    return a


def _bufs_for(q, k_pool, page_table, num_draws, bufs, team_probs=False, dense=False):
    if bufs is not None:
        return bufs
    B, Hq, d = q.shape
    _, Hkv, T, _ = k_pool.shape
    return DecodeBuffers.allocate(q.dtype, B, Hq, Hkv, d, T, page_table.shape[1], num_draws,
                                  q.device, team_probs=team_probs, dense=dense)


def santa_append_kv(k_new, v_new, k_pool, v_pool, reps, page_table, seq_lens,
                    seq_lens_next: torch.Tensor | None = None,
                    device_status: torch.Tensor | None = None, stream=None):
    """Write one new token per (sequence, KV head) (k_new, v_new [B][Hkv][d]) at position
    seq_lens[b] of the paged cache and refresh its page's representative; seq_lens_next (if
    given) receives seq_lens + 1.  All tensors on the device; nothing is allocated."""
    _req(k_new, "k_new", ndim=3)
    _req(v_new, "v_new", ndim=3)
    _req(k_pool, "k_pool", ndim=4)
    _req(reps, "reps", torch.float32, 3)
    _req(page_table, "page_table", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    if seq_lens_next is not None:
        _req(seq_lens_next, "seq_lens_next", torch.int32, 1)
    if k_new.dtype not in _DTYPES or {k_new.dtype, v_new.dtype, k_pool.dtype, v_pool.dtype} != {k_new.dtype}:
        raise SantaError("k_new, v_new, k_pool and v_pool must share one dtype")
    P, Hkv, T, d = k_pool.shape
    B = k_new.shape[0]
    if tuple(k_new.shape) != (B, Hkv, d) or tuple(v_new.shape) != (B, Hkv, d) or \
            tuple(v_pool.shape) != tuple(k_pool.shape):
        raise SantaError("k_new / v_new must be [B][Hkv][d] matching the pool")
    _check(lib().santa_append_kv(_ptr(k_new), _ptr(v_new), _DTYPES[k_new.dtype], B, Hkv, T, d,
                                 page_table.shape[1], P, _ptr(page_table), _ptr(seq_lens),
                                 _ptr(k_pool), _ptr(v_pool), _ptr(reps), _ptr(seq_lens_next),
                                 _ptr(device_status), _stream(stream)), "santa_append_kv")


def santa_sample(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws: int, seed: int,
                 bufs: DecodeBuffers | None = None, team_probs: bool = False,
                 stream=None, sampler: str = "iid_ht", mix_alpha: float = 0.0) -> DecodeBuffers:
    """Team distribution, M draws, distinct set and 1 / weight per selected team (the
    inclusion probability for the Horvitz-Thompson samplers)."""
    bufs = _bufs_for(q, k_pool, page_table, num_draws, bufs, team_probs)
    a = _args(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws, seed, bufs, sampler,
              mix_alpha)
    _check(lib().santa_sample(ctypes.byref(a), _stream(stream)), "santa_sample")
    return bufs


def santa_attend(q, k_pool, v_pool, page_table, seq_lens, sel_ids, sel_count, pi,
                 bufs: DecodeBuffers | None = None, stream=None) -> DecodeBuffers:
    """Horvitz-Thompson attention over the given teams (sel_ids [B][Hkv][M], sel_count
    [B][Hkv], pi [B][Hkv][M]); writes bufs.out."""
    _req(sel_ids, "sel_ids", torch.int32, 3)
    _req(sel_count, "sel_count", torch.int32, 2)
    _req(pi, "pi", torch.float32, 3)
    M = sel_ids.shape[2]
    bufs = _bufs_for(q, k_pool, page_table, M, bufs)
    a = _args(q, k_pool, v_pool, None, page_table, seq_lens, M, 0, bufs)
    a.sel_ids, a.sel_count, a.pi = _ptr(sel_ids), _ptr(sel_count), _ptr(pi)
    _check(lib().santa_attend(ctypes.byref(a), _stream(stream)), "santa_attend")
    return bufs


def santa_attend_vs(q, k_pool, v_pool, page_table, seq_lens, sel_ids, sel_count, pi,
                    value_rows: int, seed: int, bufs: DecodeBuffers | None = None,
                    value_ids: bool = False, stream=None):
    """Attention over the given teams with value-row sampling inside each (value_rows rows
    per team, drawn from the group-mean in-team softmax with key `seed`); writes bufs.out.
    Returns (bufs, value_ids [B][Hkv][M][value_rows] int32 or None)."""
    _req(sel_ids, "sel_ids", torch.int32, 3)
    _req(sel_count, "sel_count", torch.int32, 2)
    _req(pi, "pi", torch.float32, 3)
    B, Hq, d = q.shape
    Hkv = k_pool.shape[1]
    M = sel_ids.shape[2]
    bufs = _bufs_for(q, k_pool, page_table, M, bufs)
    need = lib().santa_attend_vs_workspace_bytes(B, Hq, Hkv, d, M)
    if need == 0:
        raise SantaError("unsupported shape for santa_attend_vs")
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    vids = (torch.empty((B, Hkv, M, value_rows), dtype=torch.int32, device=q.device)
            if value_ids else None)
    a = _args(q, k_pool, v_pool, None, page_table, seq_lens, M, seed, bufs)
    a.sel_ids, a.sel_count, a.pi = _ptr(sel_ids), _ptr(sel_count), _ptr(pi)
    a.workspace, a.workspace_bytes = _ptr(ws), need
    _check(lib().santa_attend_vs(ctypes.byref(a), value_rows, _ptr(vids), _stream(stream)),
           "santa_attend_vs")
    return bufs, vids


def santa_decode(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws: int, seed: int,
                 bufs: DecodeBuffers | None = None, team_probs: bool = False,
                 stream=None, sampler: str = "iid_ht", mix_alpha: float = 0.0) -> DecodeBuffers:
    """One SANTA++ decode step: sampling then weighted attention (Horvitz-Thompson by
    default; see SAMPLERS and the defensive mixture weight mix_alpha)."""
    bufs = _bufs_for(q, k_pool, page_table, num_draws, bufs, team_probs)
    a = _args(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws, seed, bufs, sampler,
              mix_alpha)
    _check(lib().santa_decode(ctypes.byref(a), _stream(stream)), "santa_decode")
    return bufs


def santa_decode_noalloc(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws: int,
                         seed: int, bufs: DecodeBuffers, stream=None) -> DecodeBuffers:
    """santa_decode with the library's built-in scratch instead of bufs.workspace, for
    callers that cannot allocate device memory at call time (the caller still provides the
    outputs in bufs, team_probs included if wanted; bufs.workspace is not used)."""
    a = _args(q, k_pool, v_pool, reps, page_table, seq_lens, num_draws, seed, bufs)
    _check(lib().santa_decode_noalloc(ctypes.byref(a), _stream(stream)), "santa_decode_noalloc")
    return bufs


_PLAN_MODES = {"decode": 0, "sample": 1, "attend": 2, "dense": 3}


def santa_decode_plan(q, k_pool, page_table, num_draws: int, which: str = "decode",
                      workspace_bytes: int | None = None) -> dict:
    """The launch shape the library picks: cluster size, clusters per unit, teams per CTA,
    the device's co-resident cluster count for that size, and whether the wide
    (one-CTA-per-SM) variant runs."""
    B, Hq, d = q.shape
    _, Hkv, T, _ = k_pool.shape
    a = _DecodeArgs()
    a.dtype, a.batch, a.num_q_heads, a.num_kv_heads = _DTYPES[q.dtype], B, Hq, Hkv
    a.head_dim, a.team_size, a.max_teams, a.num_draws = d, T, page_table.shape[1], num_draws
    a.num_pages = k_pool.shape[0]
    if workspace_bytes is None:
        workspace_bytes = (santa_dense_workspace_bytes(q.dtype, B, Hq, Hkv, d, T,
                                                       page_table.shape[1])
                           if which == "dense" else
                           santa_decode_workspace_bytes(q.dtype, B, Hq, Hkv, d, T,
                                                        page_table.shape[1], num_draws))
    a.workspace = 256 if workspace_bytes else None        # only its size is read
    a.workspace_bytes = workspace_bytes
    out = (ctypes.c_int32 * 5)()
    _check(lib().santa_decode_plan(ctypes.byref(a), _PLAN_MODES[which], out), "santa_decode_plan")
    return {"cluster": out[0], "clusters_per_unit": out[1], "teams_per_cta": out[2],
            "max_active_clusters": out[3], "wide": bool(out[4])}


def santa_decode_path(q, k_pool, page_table, num_draws: int, sampler: str = "iid_ht",
                      mix_alpha: float = 0.0, workspace_bytes: int | None = None) -> str:
    """"compact" or "general": the form of the decode kernel santa_decode runs for these
    shapes and sampler settings (with the default workspace unless workspace_bytes)."""
    B, Hq, d = q.shape
    _, Hkv, T, _ = k_pool.shape
    a = _DecodeArgs()
    a.dtype, a.batch, a.num_q_heads, a.num_kv_heads = _DTYPES[q.dtype], B, Hq, Hkv
    a.head_dim, a.team_size, a.max_teams, a.num_draws = d, T, page_table.shape[1], num_draws
    a.num_pages = k_pool.shape[0]
    a.sampler, a.mix_alpha = SAMPLERS[sampler], float(mix_alpha)
    if workspace_bytes is None:
        workspace_bytes = santa_decode_workspace_bytes(q.dtype, B, Hq, Hkv, d, T,
                                                       page_table.shape[1], num_draws)
    a.workspace = 256 if workspace_bytes else None        # only its size is read
    a.workspace_bytes = workspace_bytes
    rc = lib().santa_decode_path(ctypes.byref(a))
    if rc < 0:
        _check(-rc, "santa_decode_path")
    return "compact" if rc == 1 else "general"


def santa_noalloc_scratch_bytes() -> int:
    return lib().santa_noalloc_scratch_bytes()


def santa_dense_decode(q, k_pool, v_pool, page_table, seq_lens,
                       bufs: DecodeBuffers | None = None, stream=None) -> DecodeBuffers:
    """Exact dense split-K decode attention over every token (the speed reference)."""
    bufs = _bufs_for(q, k_pool, page_table, 1, bufs, dense=True)
    a = _args(q, k_pool, v_pool, None, page_table, seq_lens, 1, 0, bufs)
    _check(lib().santa_dense_decode(ctypes.byref(a), _stream(stream)), "santa_dense_decode")
    return bufs
