"""tensor_core_gemm_02_gb300: tcgen05/TMA GEMM for one GB300 (sm_103a).

The compute lives in a C-ABI shared library built from ``csrc/`` (see
``include/tcgemm.h``).  This package holds the ctypes binding (``binding``), the
build step (``build``) and the seeded workload generators (``workloads``).
Importing the package does not load the CUDA library; the first use of a
binding function does, and it raises if the library is missing.
"""
from __future__ import annotations

__all__ = [
    "gemm", "gemm_f16", "gemm_bf16", "gemm_gather_rows", "gemm_check_device_status",
    "gemm_status_string", "GemmError", "load_library",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
