"""Sparse MLA decode over an FP8 (E4M3) latent KV cache, for GB300 (sm_103a).

The decode runs in libsmd.so (hand-written CUDA, C ABI in include/smd.h);
``binding`` is its ctypes wrapper. ``inputs`` holds the seeded synthetic
workloads. Submodules load lazily so that importing ``inputs`` does not need
the CUDA library.
"""
import importlib

__all__ = ["binding", "inputs", "build", "sparse_mla_decode", "smd_plan"]


def __getattr__(name):
    if name in ("binding", "inputs", "build"):
        return importlib.import_module(f".{name}", __name__)
    if name in ("sparse_mla_decode", "smd_plan", "smd_sparse_mla_decode",
                "smd_sparse_mla_decode_ex", "smd_scale_log2", "smd_status_str", "SmdPlan",
                "SmdError"):
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
