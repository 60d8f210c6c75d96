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
