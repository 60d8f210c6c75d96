"""The seeded synthetic inputs (CPU): the recipe the workloads follow, checked against
independent computations.

- bf16 rounding is round-to-nearest-even, as torch's conversion does it.
- Heavy tokens: exactly floor(rate * N) keys per unit carry the shift 3 * qbar / |qbar|.
- Pages: paged pools use distinct in-range page ids, and page_fill matches the lengths.
- Slots past a sequence's end hold the requested fill value (NaN in the parity tests).
- Mixture keys come in runs that share a component.
- Generation-loop queries keep each head's mixture part and redraw the noise per step,
  independently of the number of steps asked for.
"""
import numpy as np
import pytest
import torch

from sampled_sparse_decode_gb300 import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-8, 8, 20000),
                        # exact ties between two bf16 neighbours, both parities
                        (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), want)
    assert W.f32_to_bf16_bits(np.array([np.nan], np.float32))[0] == 0x7FC0
    back = W.bf16_bits_to_f32(want)
    assert np.array_equal(back, torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_heavy_tokens_carry_the_query_shift():
    """tiny_f32: 1% heavy tokens.  The keys are drawn before the heavy positions, so the same
    seed without heavy tokens gives the same keys everywhere else."""
    wl = W.generate("tiny_f32", seq_len=2048)
    plain = W.generate("tiny_f32", seq_len=2048, heavy_rate=0.0)
    K, K0 = wl.k_pool[:, 0].reshape(-1, 64), plain.k_pool[:, 0].reshape(-1, 64)
    diff = K.astype(np.float64) - K0
    rows = np.nonzero(np.abs(diff).max(axis=1) > 0)[0]
    assert rows.size == int(np.floor(0.01 * 2048)) == 20
    qbar = wl.q[0].astype(np.float64).mean(axis=0)
    shift = 3.0 * qbar / np.linalg.norm(qbar)
    np.testing.assert_allclose(diff[rows], np.broadcast_to(shift, diff[rows].shape), atol=1e-5)


def test_paged_pool_and_fill():
    wl = W.generate("llama8b_paged_32k_b16_m32", seq_lens=[1000, 130, 128, 1],
                    batch=4, heavy_rate=0.0, num_pages=64, invalid_fill=float("nan"))
    T = wl.cfg.team_size
    used = [int(wl.page_table[b, i]) for b, L in enumerate(wl.seq_lens) for i in range(-(-int(L) // T))]
    assert len(set(wl.page_table.ravel().tolist())) == wl.page_table.size
    assert all(0 <= p < 64 for p in used)
    fill = np.zeros(64, np.int32)
    for b, L in enumerate(wl.seq_lens):
        for i in range(-(-int(L) // T)):
            fill[wl.page_table[b, i]] = min(T, int(L) - i * T)
    assert np.array_equal(fill, wl.page_fill)
    # slots past each sequence's end hold NaN (bf16 0x7FC0), valid slots never do
    for b, L in enumerate(wl.seq_lens):
        last = wl.page_table[b, (int(L) - 1) // T]
        c = int(L) - ((int(L) - 1) // T) * T
        assert (wl.k_pool[last, :, c:] == 0x7FC0).all() and (wl.v_pool[last, :, c:] == 0x7FC0).all()
        assert not (wl.k_pool[last, :, :c] == 0x7FC0).any()


def test_mixture_keys_come_in_runs():
    """Keys are component mean + 0.5 N(0, I), with runs of 32..512 tokens on one component:
    neighbours inside a run are close (distance about 0.5 sqrt(2 d)), keys of different
    components are far apart (about sqrt(2 d) * sqrt(1 + 0.25))."""
    wl = W.generate("qwen7b_32k_b1_m31", seq_len=4096)
    K = W.bf16_bits_to_f32(wl.k_pool[:, 0]).reshape(-1, 128).astype(np.float64)
    step = np.linalg.norm(K[1:] - K[:-1], axis=1)
    near = step < 0.5 * np.sqrt(2 * 128) * 1.3
    # a run of >= 32 tokens has >= 31 close neighbour pairs: at most 4096 / 32 run boundaries
    assert near.mean() > 1 - 1 / 32 - 0.01
    far = np.linalg.norm(K[:2048] - K[2048:], axis=1)
    assert np.median(far) > 1.3 * np.median(step)


def test_loop_queries_keep_the_mixture_part():
    cfg = W.CONFIGS["qwen7b_32k_b1_m31"]
    q5 = W.loop_queries(cfg, 5)
    assert q5.shape == (5, 1, 28, 128) and q5.dtype == np.uint16
    assert np.array_equal(W.loop_queries(cfg, 3), q5[:3])          # independent of the count
    Q = W.bf16_bits_to_f32(W.loop_queries(cfg, 400)).astype(np.float64)[:, 0]
    # per element the steps vary only by 0.3 * N(0, 1) noise around a fixed part
    assert abs(Q.std(axis=0).mean() - 0.3) < 0.01
    # that fixed part is the one the workload's own query was built from
    q = W.bf16_bits_to_f32(W.generate(cfg, seq_len=256).q).astype(np.float64)[0]
    resid = q - Q.mean(axis=0)
    assert abs(resid.std() - 0.3) < 0.02
    g = W.loop_queries(W.CONFIGS["tiny_f32"], 300)
    assert g.dtype == np.float32 and abs(g.std() - 1.0) < 0.02 and abs(g.mean()) < 0.02
