"""Seeded synthetic decode-step workloads (inputs only; none of the method's arithmetic).

Both the CUDA path and the CPU oracle consume these arrays, so this module is the one place
they share.  The shapes and value distributions stand in for the pages' evaluation setting
(Qwen2.5-7B-Instruct and Llama-3.1-8B decode attention at 32K context, "SANTA++: Sampling
Attention through Representative Keys", abstract; "Stochastic Sparse Attention for
Memory-Bound Inference", abstract): no model weights or datasets are used.

Key distributions:
  gauss    K, V, q ~ N(0, 1).
  mixture  per (sequence, KV head) 64 component means mu_c ~ N(0, I); the keys come in
           contiguous runs of U{32..512} tokens sharing a component U{0..63}, each key
           mu_c + 0.5 N(0, I); V ~ N(0, 1); query head g of the group takes 3 distinct
           components and q_g = 0.7 mean(mu) + 0.3 N(0, I).
  heavy    floor(rate * N) distinct positions per (sequence, KV head) get
           K_j += 3 qbar / |qbar|, qbar the mean of the group's query vectors.
bf16 data are rounded once, to nearest even, before either side sees them; the arrays then
hold the bf16 bit patterns as uint16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Config:
    name: str
    dtype: str          # "f32" or "bf16" (q, K and V)
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    seq_len: int        # tokens per sequence
    team_size: int      # T, also the KV page size
    draws: int          # M
    keys: str           # "gauss" or "mixture"
    heavy_rate: float   # share of "heavy" tokens
    paged: bool         # random page-table permutation over a shared pool
    num_pages: int      # pool size when paged (0: exactly the pages needed)
    data_seed: int

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def n_teams(self) -> int:
        return -(-self.seq_len // self.team_size)


CONFIGS = {
    # tiny fp32 case the oracle finishes in milliseconds
    "tiny_f32": Config("tiny_f32", "f32", 1, 2, 1, 64, 2048, 64, 8, "gauss", 0.01, False, 0, 0),
    # Qwen2.5-7B-shaped decode attention layer, one sequence, M = 31
    "qwen7b_32k_b1_m31": Config("qwen7b_32k_b1_m31", "bf16", 1, 28, 4, 128, 32768, 128, 31,
                                "mixture", 0.0, False, 0, 1),
    # the same shape with 8 independent sequences and M = 64
    "qwen7b_32k_b8_m64": Config("qwen7b_32k_b8_m64", "bf16", 8, 28, 4, 128, 32768, 128, 64,
                                "mixture", 0.0, False, 0, 2),
    # Llama-3.1-8B-shaped paged cache: 16 sequences over a shared pool of 4096 pages
    "llama8b_paged_32k_b16_m32": Config("llama8b_paged_32k_b16_m32", "bf16", 16, 32, 8, 128,
                                        32768, 128, 32, "mixture", 0.005, True, 4096, 3),
    # long context: 4 sequences of 131072 tokens (1024 teams) over a paged pool
    "long_128k_b4_m64": Config("long_128k_b4_m64", "bf16", 4, 28, 4, 128, 131072, 128, 64,
                               "mixture", 0.0, True, 4096, 4),
}


@dataclass
class Workload:
    cfg: Config
    q: np.ndarray           # [B][Hq][d] float32, or uint16 bf16 bits
    k_pool: np.ndarray      # [P][Hkv][T][d]
    v_pool: np.ndarray      # [P][Hkv][T][d]
    page_table: np.ndarray  # [B][max_teams] int32
    seq_lens: np.ndarray    # [B] int32
    page_fill: np.ndarray   # [P] int32 valid tokens per page (0 for unused pages)

    @property
    def max_teams(self) -> int:
        return self.page_table.shape[1]

    @property
    def num_pages(self) -> int:
        return self.k_pool.shape[0]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); NaN stays a quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    out = ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _unit_rng(seed: int, b: int, h: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, b, h, salt])))


def _mixture_queries(rng: np.random.Generator, mus: np.ndarray, G: int, d: int):
    """Each query head takes 3 distinct components of its KV head's mixture:
    q_g = 0.7 * mean of their means + 0.3 * N(0, I).  Returns (q, the 0.7 * mean part)."""
    q = np.empty((G, d))
    base = np.empty((G, d))
    for g in range(G):
        comps = rng.choice(64, size=3, replace=False)
        base[g] = 0.7 * mus[comps].mean(axis=0)
        q[g] = base[g] + 0.3 * rng.standard_normal(d)
    return q, base


def _gen_unit(cfg: Config, b: int, h: int, n_tok: int):
    """q [G][d], K [n_tok][d], V [n_tok][d] in float64 for unit (b, h)."""
    rng = _unit_rng(cfg.data_seed, b, h)
    G, d = cfg.group, cfg.head_dim
    if cfg.keys == "gauss":
        q = rng.standard_normal((G, d))
        K = rng.standard_normal((n_tok, d))
    elif cfg.keys == "mixture":
        mus = rng.standard_normal((64, d))
        q, _ = _mixture_queries(rng, mus, G, d)
        comp = np.empty(n_tok, dtype=np.int64)
        pos = 0
        while pos < n_tok:
            run = int(rng.integers(32, 513))
            comp[pos:pos + run] = int(rng.integers(0, 64))
            pos += run
        K = mus[comp] + 0.5 * rng.standard_normal((n_tok, d))
    else:
        raise ValueError(cfg.keys)
    n_heavy = int(np.floor(cfg.heavy_rate * n_tok))
    if n_heavy:
        qbar = q.mean(axis=0)
        where = rng.choice(n_tok, size=n_heavy, replace=False)
        K[where] += 3.0 * qbar / np.linalg.norm(qbar)
    V = rng.standard_normal((n_tok, d))
    return q, K, V


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x.astype(np.float32)
    return x32 if dtype == "f32" else f32_to_bf16_bits(x32)


def generate(cfg: Config | str, seq_lens=None, invalid_fill: float = 0.0,
             threads: int | None = None, **overrides) -> Workload:
    """Build the decode-step inputs of `cfg` (a Config or a CONFIGS name).

    seq_lens      per-sequence lengths (default: cfg.seq_len for every sequence); the
                  pages hold ceil(max(seq_lens)/T) teams per sequence.
    invalid_fill  value stored in page slots past a sequence's end (NaN is allowed).
    overrides     Config fields to replace (e.g. draws=4096, batch=2).
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    if overrides:
        cfg = replace(cfg, **overrides)
    B, Hkv, T, d = cfg.batch, cfg.kv_heads, cfg.team_size, cfg.head_dim
    lens = np.full(B, cfg.seq_len, dtype=np.int32) if seq_lens is None else \
        np.asarray(seq_lens, dtype=np.int32).copy()
    assert lens.shape == (B,) and (lens >= 1).all()
    max_teams = int(-(-int(lens.max()) // T))
    pages_needed = B * max_teams
    if cfg.paged:
        P = cfg.num_pages or pages_needed
        assert P >= pages_needed, "pool too small"
        perm = np.random.Generator(np.random.PCG64(
            np.random.SeedSequence([cfg.data_seed, 7919]))).permutation(P)
        page_table = perm[:pages_needed].reshape(B, max_teams).astype(np.int32)
    else:
        P = pages_needed
        page_table = np.arange(pages_needed, dtype=np.int32).reshape(B, max_teams)

    store_dt = np.float32 if cfg.dtype == "f32" else np.uint16
    fill_bits = _store(np.array([invalid_fill]), cfg.dtype)[0]
    k_pool = np.full((P, Hkv, T, d), fill_bits, dtype=store_dt)
    v_pool = np.full((P, Hkv, T, d), fill_bits, dtype=store_dt)
    q = np.zeros((B, cfg.q_heads, d), dtype=store_dt)
    G = cfg.group

    def work(bh):
        b, h = bh
        L = int(lens[b])
        qg, K, V = _gen_unit(cfg, b, h, L)
        q[b, h * G:(h + 1) * G] = _store(qg, cfg.dtype)
        Ks, Vs = _store(K, cfg.dtype), _store(V, cfg.dtype)
        for i in range(-(-L // T)):
            p = page_table[b, i]
            lo, hi = i * T, min((i + 1) * T, L)
            k_pool[p, h, :hi - lo] = Ks[lo:hi]
            v_pool[p, h, :hi - lo] = Vs[lo:hi]

    units = [(b, h) for b in range(B) for h in range(Hkv)]
    nthreads = threads or min(len(units), os.cpu_count() or 1, 16)
    if nthreads > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, units))
    else:
        for u in units:
            work(u)

    page_fill = np.zeros(P, dtype=np.int32)
    for b in range(B):
        L = int(lens[b])
        for i in range(-(-L // T)):
            page_fill[page_table[b, i]] = min(T, L - i * T)
    return Workload(cfg, q, k_pool, v_pool, page_table, lens, page_fill)


def loop_queries(cfg: Config | str, steps: int) -> np.ndarray:
    """Queries of a generation of `steps` tokens, [steps][B][Hq][d] in the workload's dtype.

    Each query head keeps the mixture components its step-0 query was built from and draws
    fresh noise every step: q_t = 0.7 * mean of the components + 0.3 * N(0, I) (for Gaussian
    keys, q_t ~ N(0, I)).  The noise of step t comes from its own seeded stream, so the
    sequence does not depend on how many steps are generated."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    G, d = cfg.group, cfg.head_dim
    out = np.empty((steps, cfg.batch, cfg.q_heads, d), dtype=np.float64)
    for b in range(cfg.batch):
        for h in range(cfg.kv_heads):
            if cfg.keys == "mixture":
                rng = _unit_rng(cfg.data_seed, b, h)
                _, base = _mixture_queries(rng, rng.standard_normal((64, d)), G, d)
                scale = 0.3
            else:
                base, scale = np.zeros((G, d)), 1.0
            for t in range(steps):
                noise = _unit_rng(cfg.data_seed, b, h, salt=1 + t).standard_normal((G, d))
                out[t, b, h * G:(h + 1) * G] = base + scale * noise
    return _store(out, cfg.dtype)
