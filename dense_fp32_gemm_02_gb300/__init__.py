"""GB300-native FP32 SGEMM: C = alpha*A*B + beta*C, row-major, behind a C ABI.

The compute path is ``libsgemm`` (hand-written CUDA for sm_103a, built from
``csrc/``); ``binding`` marshals torch tensors to it and nothing else.  The
binding is imported lazily so that the seeded input generators in
``workloads`` can be used without the CUDA library; calling any SGEMM entry
point without a built library raises immediately (there is no CPU fallback).
"""

__all__ = ["sgemm", "sgemm_host", "sgemm_into", "library_path", "workloads"]


def __getattr__(name):
    if name in ("sgemm", "sgemm_host", "sgemm_into", "library_path", "lib"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
