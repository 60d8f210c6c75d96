"""The C ABI without a GPU: libsanta.so builds for sm_103a, loads, exports every function
include/santa.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from sampled_sparse_decode_gb300 import build as B
from sampled_sparse_decode_gb300.binding import _DecodeArgs

HEADER = os.path.join(B.INCLUDE, "santa.h")
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(B.build())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(santa_\w+)\s*\(", text, re.M)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10, names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in santa.h but not exported"


def test_version_and_status_strings(lib):
    lib.santa_abi_version.restype = ctypes.c_int
    assert lib.santa_abi_version() == 1
    lib.santa_status_string.restype = ctypes.c_char_p
    for s in range(5):
        assert lib.santa_status_string(s)
    assert b"unknown" in lib.santa_status_string(99)


def valid_args():
    a = _DecodeArgs()
    fake = 0x10000  # 16-byte-aligned, never dereferenced: every call below fails its checks first
    for f in ("q", "k_pool", "v_pool", "reps", "page_table", "seq_lens", "out", "draw_ids",
              "sel_ids", "sel_count", "pi", "device_status"):
        setattr(a, f, fake)
    a.dtype, a.batch, a.num_q_heads, a.num_kv_heads = 1, 1, 28, 4
    a.head_dim, a.team_size, a.max_teams, a.num_draws = 128, 128, 256, 31
    a.num_pages, a.seed = 256, 0
    return a


@pytest.mark.parametrize("field,value,expect", [
    ("dtype", 7, UNSUPPORTED), ("head_dim", 96, UNSUPPORTED), ("team_size", 32, UNSUPPORTED),
    ("num_q_heads", 36, UNSUPPORTED), ("num_q_heads", 30, INVALID), ("num_draws", 0, UNSUPPORTED),
    ("num_draws", 5000, UNSUPPORTED), ("max_teams", 20000, UNSUPPORTED), ("batch", 0, INVALID),
    ("num_pages", 0, INVALID), ("q", 0, INVALID), ("q", 0x10008, INVALID), ("sel_ids", 0, INVALID),
    ("reps", 0, INVALID), ("sampler", 3, INVALID), ("sampler", -1, INVALID),
    ("mix_alpha", -0.25, INVALID), ("mix_alpha", 1.5, INVALID), ("mix_alpha", float("nan"), INVALID),
])
def test_sample_rejects_bad_arguments_on_host(lib, field, value, expect):
    a = valid_args()
    setattr(a, field, value)
    lib.santa_sample.restype = ctypes.c_int
    assert lib.santa_sample(ctypes.byref(a), None) == expect


def test_null_args(lib):
    for fn in ("santa_sample", "santa_attend", "santa_decode", "santa_dense_decode",
               "santa_decode_noalloc"):
        getattr(lib, fn).restype = ctypes.c_int
        assert getattr(lib, fn)(None, None) == INVALID
    a = valid_args()
    a.out = 0
    assert lib.santa_attend(ctypes.byref(a), None) == INVALID
    assert lib.santa_decode(ctypes.byref(a), None) == INVALID


def test_host_step_rejects_missing_buffers(lib):
    f = lib.santa_decode_host
    f.restype = ctypes.c_int
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    f.argtypes = [ctypes.c_void_p, vp, vp, sz, vp, vp, sz, vp]
    a = valid_args()
    assert f(None, 0x1000, 0x2000, 16, 0x3000, 0x4000, 16, None) == INVALID
    assert f(ctypes.addressof(a), None, 0x2000, 16, 0x3000, 0x4000, 16, None) == INVALID
    assert f(ctypes.addressof(a), 0x1000, None, 16, 0x3000, 0x4000, 16, None) == INVALID
    assert f(ctypes.addressof(a), 0x1000, 0x2000, 16, None, 0x4000, 16, None) == INVALID
    assert f(ctypes.addressof(a), 0x1000, 0x2000, 16, 0x3000, None, 16, None) == INVALID


def test_host_copy_route_without_device_memory(lib):
    # null pointers, no bytes, unaligned sizes and plain (not page-locked) host memory all
    # take the copy engine; nothing is enqueued either way
    f = lib.santa_host_copy_route
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
    buf = (ctypes.c_ubyte * 4096)()
    host = (ctypes.addressof(buf) + 15) // 16 * 16
    assert f(None, 0x2000, 64) == 0
    assert f(host, None, 64) == 0
    assert f(host, 0x2000, 0) == 0
    assert f(host, 0x2000, 24) == 0
    assert f(host, 0x2000, 64) == 0


def test_reps_reject_bad_arguments_on_host(lib):
    f = lib.santa_build_reps
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert f(0x10000, 2, 16, 4, 128, 128, None, 0x20000, None, None) == UNSUPPORTED
    assert f(0x10000, 1, 16, 4, 128, 100, None, 0x20000, None, None) == UNSUPPORTED
    assert f(None, 1, 16, 4, 128, 128, None, 0x20000, None, None) == INVALID
    assert f(0x10000, 1, 0, 4, 128, 128, None, 0x20000, None, None) == INVALID


def test_minimum_workspace_size(lib):
    f = lib.santa_decode_workspace_min_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 7
    # a unit needs scratch only when it spans several clusters: with 16-CTA clusters of at
    # most 256 chunks (64 tokens) each, 31 draws over 256 teams fit one cluster
    assert f(1, 28, 4, 128, 128, 256, 31) == 256
    # 4096 draws of 128-token teams: 8192 chunks -> 2 clusters; 256 slack + counters (256)
    # + (m, l) [4][2][7][2] fp32 rounded to 256 + acc [4][2][7][128] fp32
    assert f(1, 28, 4, 128, 128, 16384, 4096) == 256 + 256 + 512 + 4 * 2 * 7 * 128 * 4
    assert f(1, 30, 4, 128, 128, 256, 31) == 0


SCRATCH_LIMIT = 5


def test_append_rejects_bad_arguments_on_host(lib):
    f = lib.santa_append_kv
    f.restype = ctypes.c_int
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    good = dict(k_new=0x10000, v_new=0x20000, dtype=1, batch=2, hkv=4, T=128, d=128, mt=256,
                P=512, pt=0x30000, lens=0x40000, k=0x50000, v=0x60000, reps=0x70000,
                nxt=0x80000, status=0x90000)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["k_new"], a["v_new"], a["dtype"], a["batch"], a["hkv"], a["T"], a["d"],
                 a["mt"], a["P"], a["pt"], a["lens"], a["k"], a["v"], a["reps"], a["nxt"],
                 a["status"], None)

    assert call(dtype=7) == UNSUPPORTED
    assert call(d=96) == UNSUPPORTED
    assert call(T=32) == UNSUPPORTED
    assert call(mt=20000) == UNSUPPORTED
    assert call(batch=0) == INVALID
    assert call(P=0) == INVALID
    assert call(k_new=None) == INVALID
    assert call(reps=None) == INVALID
    assert call(k=0x50008) == INVALID                    # not 16-byte aligned
    assert call(pt=0x30002) == INVALID
    assert call(nxt=0x40000) == INVALID                  # lengths written while read


def test_update_reps_needs_a_page_list(lib):
    f = lib.santa_update_reps
    f.restype = ctypes.c_int
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [vp, i32, i64, i32, i32, i32, vp, i32, vp, vp, vp, vp]
    assert f(0x10000, 1, 16, 4, 128, 128, None, 3, None, 0x20000, None, None) == INVALID
    assert f(0x10000, 1, 16, 4, 128, 128, 0x30002, 3, None, 0x20000, None, None) == INVALID


def test_value_sampling_rejects_bad_arguments_on_host(lib):
    f = lib.santa_attend_vs
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    ws = lib.santa_attend_vs_workspace_bytes
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int] * 5
    a = valid_args()
    need = ws(a.batch, a.num_q_heads, a.num_kv_heads, a.head_dim, a.num_draws)
    assert need > 0
    a.workspace, a.workspace_bytes = 0xA0000, need - 1
    assert f(ctypes.byref(a), 16, None, None) == INVALID          # workspace one byte short
    for rows in (0, 257):
        assert f(ctypes.byref(a), rows, None, None) == UNSUPPORTED
    a.num_draws = 2000
    assert f(ctypes.byref(a), 16, None, None) == UNSUPPORTED
    a = valid_args()
    a.workspace, a.workspace_bytes = 0xA0000, need
    a.out = 0x10008                                                 # out must be 16-byte aligned
    assert f(ctypes.byref(a), 16, None, None) == INVALID
    a = valid_args()
    a.workspace, a.workspace_bytes = 0xA0000, need
    assert f(ctypes.byref(a), 16, 0x30002, None) == INVALID         # value_ids misaligned
    assert f(None, 16, None, None) == INVALID


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    f = lib.santa_decode_noalloc
    f.restype = ctypes.c_int
    lib.santa_noalloc_scratch_bytes.restype = ctypes.c_size_t
    assert lib.santa_noalloc_scratch_bytes() == 4 << 20
    a = valid_args()
    a.head_dim = 96
    assert f(ctypes.byref(a), None) == UNSUPPORTED
    # 4096 draws of 128-token teams over 16384 teams, 64 sequences x 8 heads: the split
    # partials alone exceed the 4 MiB scratch
    a = valid_args()
    a.batch, a.num_q_heads, a.num_kv_heads, a.max_teams, a.num_draws = 64, 64, 8, 16384, 4096
    assert f(ctypes.byref(a), None) == SCRATCH_LIMIT
    # one cluster per unit (M = 1), so the split partials need nothing, but 65535 x 32
    # units' arrival counters (8 MiB) would not fit: refused before any CUDA call
    a = valid_args()
    a.batch, a.num_q_heads, a.num_kv_heads, a.num_draws = 65535, 32, 32, 1
    assert f(ctypes.byref(a), None) == SCRATCH_LIMIT
    # the largest unit count whose counters still fit passes the size checks (the call then
    # fails on something else: no device here, or, on a GPU, the misaligned query, which is
    # refused before the array is touched)
    units_max = ((4 << 20) - 256) // 4
    a = valid_args()
    a.batch, a.num_q_heads, a.num_kv_heads, a.num_draws = units_max // 16, 16, 16, 1
    lib.santa_decode_workspace_min_bytes.restype = ctypes.c_size_t
    assert lib.santa_decode_workspace_min_bytes(a.batch, 16, 16, 128, 128, 256, 1) <= 4 << 20
    a.q = 0x10008
    assert f(ctypes.byref(a), None) != SCRATCH_LIMIT
