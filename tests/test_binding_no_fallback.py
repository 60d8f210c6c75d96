"""No CPU fallback (CPU): every public call of the binding refuses tensors that are not on a
CUDA device with a SantaError, before anything is computed.  The product path has no CPU
implementation to fall back to."""
import pytest
import torch

import sampled_sparse_decode_gb300 as santa
from sampled_sparse_decode_gb300.binding import SantaError

B, Hq, Hkv, d, T, P, M = 1, 4, 2, 64, 64, 8, 4


def _inputs():
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16)
    k = torch.zeros(P, Hkv, T, d, dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    reps = torch.zeros(P, Hkv, d, dtype=torch.float32)
    pt = torch.arange(P, dtype=torch.int32).view(B, P)
    lens = torch.full((B,), 100, dtype=torch.int32)
    return q, k, v, reps, pt, lens


CALLS = {
    "santa_build_reps": lambda q, k, v, r, pt, L: santa.santa_build_reps(k),
    "santa_update_reps": lambda q, k, v, r, pt, L: santa.santa_update_reps(
        k, torch.zeros(1, dtype=torch.int32), r),
    "santa_append_kv": lambda q, k, v, r, pt, L: santa.santa_append_kv(
        q[:, :Hkv].contiguous(), q[:, :Hkv].contiguous(), k, v, r, pt, L),
    "santa_sample": lambda q, k, v, r, pt, L: santa.santa_sample(q, k, v, r, pt, L, M, 0),
    "santa_attend": lambda q, k, v, r, pt, L: santa.santa_attend(
        q, k, v, pt, L, torch.zeros(B, Hkv, M, dtype=torch.int32),
        torch.ones(B, Hkv, dtype=torch.int32), torch.ones(B, Hkv, M)),
    "santa_decode": lambda q, k, v, r, pt, L: santa.santa_decode(q, k, v, r, pt, L, M, 0),
    "santa_dense_decode": lambda q, k, v, r, pt, L: santa.santa_dense_decode(q, k, v, pt, L),
    "santa_attend_vs": lambda q, k, v, r, pt, L: santa.santa_attend_vs(
        q, k, v, pt, L, torch.zeros(B, Hkv, M, dtype=torch.int32),
        torch.ones(B, Hkv, dtype=torch.int32), torch.ones(B, Hkv, M), 8, 0),
    "santa_decode_prepared": lambda q, k, v, r, pt, L: santa.santa_decode_prepared(
        q, k, v, r, pt, L, M),
}


@pytest.mark.parametrize("name", list(CALLS))
def test_cpu_tensors_are_refused(name):
    with pytest.raises(SantaError):
        CALLS[name](*_inputs())
