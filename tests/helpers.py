"""Shared helpers of the test suite: device copies of seeded workloads, oracle problems,
and the parity rules (tolerances and the CDF-boundary window for draw mismatches)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from sampled_sparse_decode_gb300 import workloads as W

# Output tolerances (max-abs), for outputs computed on identical sampled sets: fp32 inputs
# with fp32 arithmetic, and bf16 inputs with fp32 accumulation.
TOL_OUT = {"f32": 1e-5, "bf16": 2e-3}
# A draw may differ from the oracle's only if the oracle's u*Z lies this close (relative to
# Z) to one of the oracle's CDF values (the team probabilities come from fp32 scores on the
# GPU and fp64 ones in the oracle; the decision itself is exact integer arithmetic on both) ...
BOUNDARY_WINDOW = 1e-6
# ... and such draws must stay below this share of all draws.
BOUNDARY_SHARE = 1e-4
# Relative tolerance of the inclusion probabilities.
TOL_PI = 1e-5


def problem(wl: W.Workload) -> oracle.Problem:
    return oracle.Problem(wl.q, wl.k_pool, wl.v_pool, wl.page_table, wl.seq_lens)


def to_torch(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceWorkload:
    """A workload's inputs on the GPU (q, k_pool, v_pool, page_table, seq_lens, page_fill)."""

    def __init__(self, wl: W.Workload, device="cuda"):
        self.wl = wl
        self.q = to_torch(wl.q, device)
        self.k_pool = to_torch(wl.k_pool, device)
        self.v_pool = to_torch(wl.v_pool, device)
        self.page_table = to_torch(wl.page_table, device)
        self.seq_lens = to_torch(wl.seq_lens, device)
        self.page_fill = to_torch(wl.page_fill, device)


@functools.lru_cache(maxsize=2)
def full_workload(name: str) -> W.Workload:
    return W.generate(name)


@functools.lru_cache(maxsize=2)
def full_oracle_reps(name: str) -> np.ndarray:
    wl = full_workload(name)
    return oracle.build_reps(problem(wl), wl.page_fill)


def boundary_distance(t: int, C: np.ndarray) -> float:
    """Distance from the draw point t to the nearest CDF value (an interval boundary), in
    units of the CDF total Z (t and C are the oracle's fixed-point integers)."""
    if not C.size:
        return float("inf")
    Cf = C.astype(np.float64)
    return float(np.min(np.abs(Cf - float(t)))) / float(Cf[-1])


def compare_draws(gpu_draws: np.ndarray, ora_draws: np.ndarray, t: np.ndarray, C: np.ndarray):
    """Returns (mismatches inside the boundary window, mismatches outside it)."""
    inside = outside = 0
    for r in np.nonzero(gpu_draws != ora_draws)[0]:
        if boundary_distance(int(t[r]), C) <= BOUNDARY_WINDOW:
            inside += 1
        else:
            outside += 1
    return inside, outside
