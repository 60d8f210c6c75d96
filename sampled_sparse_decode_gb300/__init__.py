"""SANTA++ decode-step attention on GB300 (sm_103a): a C-ABI CUDA library and its binding.

``santa_build_reps``, ``santa_update_reps``, ``santa_append_kv``, ``santa_sample``,
``santa_attend``, ``santa_decode`` and ``santa_dense_decode`` call the entry points of ``libsanta.so`` with
torch CUDA tensors; every step of the path runs in that library's kernels.  The library is
loaded on first use and a missing or unbuildable library raises an error: there is no CPU
fallback.  ``workloads`` builds seeded synthetic inputs and can be imported without a GPU.
"""
from __future__ import annotations

_BINDING_NAMES = (
    "santa_build_reps", "santa_update_reps", "santa_sample", "santa_attend", "santa_decode",
    "santa_dense_decode", "santa_decode_workspace_bytes", "santa_decode_workspace_min_bytes",
    "santa_dense_workspace_bytes", "santa_abi_version", "santa_status_string", "DecodeBuffers",
    "santa_decode_noalloc", "santa_noalloc_scratch_bytes", "santa_decode_plan", "santa_decode_path",
    "SantaError", "DEV_BAD_PAGE", "DEV_BAD_SEQLEN", "DEV_BAD_SEL", "santa_append_kv", "SAMPLERS",
    "santa_attend_vs", "StepInputs", "HostOutputs", "PreparedDecode", "santa_decode_prepared",
)

__all__ = list(_BINDING_NAMES) + ["workloads"]


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
