"""ctypes front end of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (``sampled_sparse_decode_gb300``) never
does, and nothing here imports the product path.

Each wrapper takes numpy arrays laid out as the pages' decode step needs them
(q [B][Hq][d], k_pool / v_pool [P][Hkv][T][d] as float32 or as bf16 bit patterns in uint16,
page_table [B][max_teams], seq_lens [B]) and returns float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no FP contraction, fp64 throughout)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
             "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("dtype", ctypes.c_int),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("num_pages", ctypes.c_int64),
        ("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("team_size", ctypes.c_int), ("max_teams", ctypes.c_int),
    ]


_lib = None


def lib():
    """The oracle library: liboracle.so, or the library named by ORACLE_LIB (the mutation
    tests load deliberately broken builds of oracle.c that way, to show the pins catch them)."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        P = ctypes.POINTER(_Problem)
        vp, i32, i64, u64, dbl = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                  ctypes.c_uint64, ctypes.c_double)
        sig = {
            "oracle_philox4x32_10": (None, [vp, vp, vp]),
            "oracle_uniform": (dbl, [u64, i32, i32, i32]),
            "oracle_elem": (dbl, [vp, i32, i64]),
            "oracle_build_reps": (i32, [P, vp, vp]),
            "oracle_team_probs": (i32, [P, vp, i32, i32, vp, vp]),
            "oracle_cdf_search": (i32, [vp, i32, u64]),
            "oracle_fixed_prob": (u64, [dbl]),
            "oracle_draw_point": (u64, [u64, i32, i32, i32, u64]),
            "oracle_draw": (None, [vp, i32, i32, u64, i32, i32, vp, vp, vp]),
            "oracle_select": (i32, [vp, i32, vp, i32, vp, vp]),
            "oracle_num_den": (i32, [P, i32, i32, vp, vp, i32, vp, vp, vp]),
            "oracle_attend": (i32, [P, i32, i32, vp, vp, i32, vp]),
            "oracle_dense": (i32, [P, i32, i32, vp]),
            "oracle_decode": (i32, [P, vp, i32, u64, i32, i32, vp, vp, vp, vp, vp]),
            "oracle_mix": (None, [vp, i32, dbl, vp]),
            "oracle_vs_row_probs": (i32, [P, i32, i32, i32, vp]),
            "oracle_vs_point": (u64, [u64, i32, i32, i32, i32, u64]),
            "oracle_vs_draw": (i32, [P, i32, i32, i32, i32, u64, vp, vp, vp]),
            "oracle_num_den_vs": (i32, [P, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp]),
            "oracle_attend_vs": (i32, [P, i32, i32, vp, vp, i32, i32, u64, vp, vp]),
            "oracle_systematic_point": (u64, [u64, i32, i32, u64]),
            "oracle_draw_systematic": (None, [vp, i32, i32, u64, i32, i32, vp, vp, vp]),
            "oracle_select_ex": (i32, [vp, i32, vp, i32, i32, vp, vp]),
            "oracle_decode_ex": (i32, [P, vp, i32, u64, i32, i32, i32, dbl, vp, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


@dataclass
class Problem:
    """One decode step's inputs, held as numpy arrays (kept alive by this object)."""
    q: np.ndarray            # [B][Hq][d] float32, or uint16 bf16 bit patterns
    k_pool: np.ndarray       # [P][Hkv][T][d]
    v_pool: np.ndarray       # [P][Hkv][T][d]
    page_table: np.ndarray   # [B][max_teams] int32
    seq_lens: np.ndarray     # [B] int32

    def __post_init__(self):
        self.dtype = BF16 if self.k_pool.dtype == np.uint16 else F32
        assert self.q.dtype == self.k_pool.dtype == self.v_pool.dtype
        self.q = np.ascontiguousarray(self.q)
        self.k_pool = np.ascontiguousarray(self.k_pool)
        self.v_pool = np.ascontiguousarray(self.v_pool)
        self.page_table = np.ascontiguousarray(self.page_table, dtype=np.int32)
        self.seq_lens = np.ascontiguousarray(self.seq_lens, dtype=np.int32)
        B, Hq, d = self.q.shape
        P, Hkv, T, d2 = self.k_pool.shape
        assert d == d2 and Hq % Hkv == 0
        self.B, self.Hq, self.Hkv, self.d, self.T, self.P = B, Hq, Hkv, d, T, P
        self.G = Hq // Hkv
        self.max_teams = self.page_table.shape[1]
        self._c = _Problem(_ptr(self.q), _ptr(self.k_pool), _ptr(self.v_pool), self.dtype,
                           _ptr(self.page_table), _ptr(self.seq_lens), P, B, Hq, Hkv, d, T,
                           self.max_teams)

    def n_teams(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.T)


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise ValueError(f"oracle {what} failed with code {rc}")
    return rc


def philox4x32_10(counter, key) -> np.ndarray:
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, b: int, h: int, r: int) -> float:
    return lib().oracle_uniform(seed, b, h, r)


def elem_values(arr: np.ndarray) -> np.ndarray:
    """The oracle's own decoding of stored elements to float64 (bf16 or float32)."""
    a = np.ascontiguousarray(arr).reshape(-1)
    dt = BF16 if a.dtype == np.uint16 else F32
    f = lib().oracle_elem
    return np.array([f(_ptr(a), dt, i) for i in range(a.size)], dtype=np.float64)


def build_reps(pr: Problem, page_fill: np.ndarray | None = None) -> np.ndarray:
    reps = np.zeros((pr.P, pr.Hkv, pr.d), dtype=np.float64)
    fill = None if page_fill is None else np.ascontiguousarray(page_fill, dtype=np.int32)
    _check(lib().oracle_build_reps(ctypes.byref(pr._c), _ptr(fill), _ptr(reps)), "build_reps")
    return reps


def team_probs(pr: Problem, reps: np.ndarray, b: int, h: int, with_scores: bool = False):
    p = np.zeros(pr.max_teams, dtype=np.float64)
    s = np.zeros((pr.G, pr.max_teams), dtype=np.float64) if with_scores else None
    n = _check(lib().oracle_team_probs(ctypes.byref(pr._c), _ptr(reps), b, h, _ptr(s), _ptr(p)),
               "team_probs")
    return (p[:n], s[:, :n]) if with_scores else p[:n]


def cdf_search(C: np.ndarray, t: int) -> int:
    C = np.ascontiguousarray(C, dtype=np.uint64)
    return lib().oracle_cdf_search(_ptr(C), C.size, int(t))


def fixed_prob(p: float) -> int:
    return int(lib().oracle_fixed_prob(float(p)))


def draw_point(seed: int, b: int, h: int, r: int, Z: int) -> int:
    return int(lib().oracle_draw_point(seed, b, h, r, int(Z)))


def draw(p: np.ndarray, M: int, seed: int, b: int, h: int):
    """Returns (draws [M] int32, t = floor(u*Z) [M] uint64, C [n] uint64), with C the
    fixed-point (2^62) integer CDF."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    n = p.size
    draws = np.zeros(M, dtype=np.int32)
    t = np.zeros(M, dtype=np.uint64)
    C = np.zeros(n, dtype=np.uint64)
    lib().oracle_draw(_ptr(p), n, M, seed, b, h, _ptr(draws), _ptr(t), _ptr(C))
    return draws, t, C


def select(draws: np.ndarray, p: np.ndarray):
    """Returns (sel ascending int32 [|S|], pi float64 [|S|])."""
    draws = np.ascontiguousarray(draws, dtype=np.int32)
    p = np.ascontiguousarray(p, dtype=np.float64)
    sel = np.zeros(max(draws.size, 1), dtype=np.int32)
    pi = np.zeros(max(draws.size, 1), dtype=np.float64)
    cnt = lib().oracle_select(_ptr(draws), draws.size, _ptr(p), p.size, _ptr(sel), _ptr(pi))
    return sel[:cnt].copy(), pi[:cnt].copy()


def num_den(pr: Problem, b: int, h: int, sel, pi, shift):
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    pi = np.ascontiguousarray(pi, dtype=np.float64)
    shift = np.ascontiguousarray(np.broadcast_to(np.asarray(shift, np.float64), (pr.G,)))
    num = np.zeros((pr.G, pr.d), dtype=np.float64)
    den = np.zeros(pr.G, dtype=np.float64)
    _check(lib().oracle_num_den(ctypes.byref(pr._c), b, h, _ptr(sel), _ptr(pi), sel.size,
                                _ptr(shift), _ptr(num), _ptr(den)), "num_den")
    return num, den


def attend(pr: Problem, b: int, h: int, sel, pi) -> np.ndarray:
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    pi = np.ascontiguousarray(pi, dtype=np.float64)
    out = np.zeros((pr.G, pr.d), dtype=np.float64)
    _check(lib().oracle_attend(ctypes.byref(pr._c), b, h, _ptr(sel), _ptr(pi), sel.size,
                               _ptr(out)), "attend")
    return out


def dense(pr: Problem, b: int, h: int) -> np.ndarray:
    out = np.zeros((pr.G, pr.d), dtype=np.float64)
    _check(lib().oracle_dense(ctypes.byref(pr._c), b, h, _ptr(out)), "dense")
    return out


@dataclass
class UnitResult:
    draws: np.ndarray   # [M] int32
    sel: np.ndarray     # [|S|] int32
    pi: np.ndarray      # [|S|] float64
    p: np.ndarray       # [n] float64
    out: np.ndarray     # [G][d] float64


def decode(pr: Problem, reps: np.ndarray, M: int, seed: int, b: int, h: int) -> UnitResult:
    draws = np.zeros(M, dtype=np.int32)
    sel = np.zeros(M, dtype=np.int32)
    pi = np.zeros(M, dtype=np.float64)
    p = np.zeros(pr.max_teams, dtype=np.float64)
    out = np.zeros((pr.G, pr.d), dtype=np.float64)
    cnt = _check(lib().oracle_decode(ctypes.byref(pr._c), _ptr(reps), M, seed, b, h,
                                     _ptr(draws), _ptr(sel), _ptr(pi), _ptr(p), _ptr(out)),
                 "decode")
    return UnitResult(draws, sel[:cnt].copy(), pi[:cnt].copy(), p[:pr.n_teams(b)].copy(), out)


# ---------------------------------------------------------------- sampler variants

SAMPLERS = {"iid_ht": 0, "systematic": 1, "iid_hh": 2}


def mix(p: np.ndarray, alpha: float) -> np.ndarray:
    """Defensive mixture q = (1 - alpha) p + alpha / n."""
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.zeros_like(p)
    lib().oracle_mix(_ptr(p), p.size, float(alpha), _ptr(q))
    return q


def systematic_point(t_u: int, r: int, M: int, Z: int) -> int:
    return int(lib().oracle_systematic_point(int(t_u), int(r), int(M), int(Z)))


def draw_systematic(q: np.ndarray, M: int, seed: int, b: int, h: int):
    """Returns (draws [M] int32, t [M] uint64, C [n] uint64) for the systematic sampler."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    n = q.size
    draws = np.zeros(M, dtype=np.int32)
    t = np.zeros(M, dtype=np.uint64)
    C = np.zeros(n, dtype=np.uint64)
    lib().oracle_draw_systematic(_ptr(q), n, M, seed, b, h, _ptr(draws), _ptr(t), _ptr(C))
    return draws, t, C


def draw_with(sampler: str, q: np.ndarray, M: int, seed: int, b: int, h: int):
    return draw_systematic(q, M, seed, b, h) if sampler == "systematic" else draw(q, M, seed, b, h)


def select_ex(draws: np.ndarray, q: np.ndarray, sampler: str):
    """Returns (sel ascending int32, recip = 1 / weight float64)."""
    draws = np.ascontiguousarray(draws, dtype=np.int32)
    q = np.ascontiguousarray(q, dtype=np.float64)
    sel = np.zeros(max(draws.size, 1), dtype=np.int32)
    rc = np.zeros(max(draws.size, 1), dtype=np.float64)
    cnt = _check(lib().oracle_select_ex(_ptr(draws), draws.size, _ptr(q), q.size,
                                        SAMPLERS[sampler], _ptr(sel), _ptr(rc)), "select_ex")
    return sel[:cnt].copy(), rc[:cnt].copy()


def decode_ex(pr: Problem, reps: np.ndarray, M: int, seed: int, b: int, h: int,
              sampler: str = "iid_ht", alpha: float = 0.0) -> UnitResult:
    """One unit's decode step with a sampler variant and defensive mixture; UnitResult.p
    holds the sampling distribution q and UnitResult.pi the 1 / weight of each team."""
    draws = np.zeros(M, dtype=np.int32)
    sel = np.zeros(M, dtype=np.int32)
    rc = np.zeros(M, dtype=np.float64)
    q = np.zeros(pr.max_teams, dtype=np.float64)
    out = np.zeros((pr.G, pr.d), dtype=np.float64)
    cnt = _check(lib().oracle_decode_ex(ctypes.byref(pr._c), _ptr(reps), M, seed, b, h,
                                        SAMPLERS[sampler], float(alpha), _ptr(draws), _ptr(sel),
                                        _ptr(rc), _ptr(q), _ptr(out)), "decode_ex")
    return UnitResult(draws, sel[:cnt].copy(), rc[:cnt].copy(), q[:pr.n_teams(b)].copy(), out)


# ---------------------------------------------------------------- value-row sampling

def vs_row_probs(pr: Problem, b: int, h: int, team: int) -> np.ndarray:
    """Group-mean in-team distribution r over the team's valid tokens."""
    r = np.zeros(pr.T, dtype=np.float64)
    n = _check(lib().oracle_vs_row_probs(ctypes.byref(pr._c), b, h, team, _ptr(r)), "vs_row_probs")
    return r[:n].copy()


def vs_draw(pr: Problem, b: int, h: int, team: int, S: int, seed: int):
    """Returns (idx [S] int32, t [S] uint64, C [len] uint64) for the row draws of a team."""
    idx = np.zeros(S, dtype=np.int32)
    t = np.zeros(S, dtype=np.uint64)
    C = np.zeros(pr.T, dtype=np.uint64)
    n = _check(lib().oracle_vs_draw(ctypes.byref(pr._c), b, h, team, S, seed, _ptr(idx), _ptr(t),
                                    _ptr(C)), "vs_draw")
    return idx, t, C[:n].copy()


def num_den_vs(pr: Problem, b: int, h: int, sel, pi, S: int, idx, shift):
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    pi = np.ascontiguousarray(pi, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1)
    shift = np.ascontiguousarray(np.broadcast_to(np.asarray(shift, np.float64), (pr.G,)))
    num = np.zeros((pr.G, pr.d), dtype=np.float64)
    den = np.zeros(pr.G, dtype=np.float64)
    _check(lib().oracle_num_den_vs(ctypes.byref(pr._c), b, h, _ptr(sel), _ptr(pi), sel.size, S,
                                   _ptr(idx), _ptr(shift), _ptr(num), _ptr(den)), "num_den_vs")
    return num, den


def attend_vs(pr: Problem, b: int, h: int, sel, pi, S: int, seed: int):
    """Returns (out [G][d], idx [|S|][S]) of the value-sampled estimate."""
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    pi = np.ascontiguousarray(pi, dtype=np.float64)
    idx = np.zeros((max(sel.size, 1), S), dtype=np.int32)
    out = np.zeros((pr.G, pr.d), dtype=np.float64)
    _check(lib().oracle_attend_vs(ctypes.byref(pr._c), b, h, _ptr(sel), _ptr(pi), sel.size, S,
                                  seed, _ptr(idx), _ptr(out)), "attend_vs")
    return out, idx[:sel.size].copy()
