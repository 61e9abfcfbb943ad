"""The allocation-free skinny entry point (gemm_skinny_noalloc) on the GPU.

This entry point is for callers that cannot call cudaMalloc where they run the
GEMM (their device memory belongs to another allocator, or they are in a
section where cudaMalloc's implicit synchronisation is not allowed).  It keeps
its scratch in a fixed array inside the library instead.  Here it is called
through the C ABI and its output is compared with gemm_bf16's on the same
inputs, within the parity tolerance, on two calls in a row (the second call
finds the array as the first one left it).

The file name makes pytest collect it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_F32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tolerance_ok(got, ref_d, A, B):
    """|got - ref| <= 2e-3 * (|A| |B|^T) + 1e-5, the bound the parity tests use."""
    absprod = A.abs().double() @ B.abs().double().T
    err = (got.double() - ref_d.double()).abs()
    return bool(torch.all(err <= 2e-3 * absprod + 1e-5))


def test_noalloc_matches_gemm_bf16_twice():
    p = workloads.random_problem(41, 16, 28672, 4096, dtype="bf16", with_c=True, alpha=0.5,
                                 beta=1.0, b_scale=0.02)
    A, B, C = p.A.to(DEV), p.B.to(DEV), p.C.to(DEV)
    lib = binding.load_library()
    stream = torch.cuda.current_stream().cuda_stream

    ref = binding.gemm_bf16(A, B, C, alpha=p.alpha, beta=p.beta, out=OUT_F32)
    assert binding.gemm_check_device_status() == binding.GEMM_OK

    D = torch.empty((p.M, p.N), dtype=torch.float32, device=DEV)
    for call in range(2):
        D.fill_(float("nan"))
        st = lib.gemm_skinny_noalloc(p.M, p.N, p.K, 1, A.data_ptr(), A.stride(0), B.data_ptr(),
                                     B.stride(0), C.data_ptr(), C.stride(0), D.data_ptr(),
                                     D.stride(0), OUT_F32, ctypes.c_float(p.alpha),
                                     ctypes.c_float(p.beta), ctypes.c_void_p(stream))
        assert st == binding.GEMM_OK, binding.gemm_status_string(st)
        assert binding.gemm_check_device_status() == binding.GEMM_OK
        assert not torch.isnan(D).any(), f"call {call}"
        assert _tolerance_ok(D.cpu(), ref.cpu(), p.A.float(), p.B.float()), f"call {call}"


def _call(lib, M, N, K, A, B, D, stream):
    return lib.gemm_skinny_noalloc(M, N, K, 1, A.data_ptr(), A.stride(0), B.data_ptr(),
                                   B.stride(0), None, 0, D.data_ptr(), D.stride(0), OUT_F32,
                                   ctypes.c_float(1.0), ctypes.c_float(0.0), stream)


def test_noalloc_rejects_what_it_cannot_hold():
    """Problems the fixed array cannot hold are refused before anything is launched
    (real buffers of the full size are passed all the same)."""
    lib = binding.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # M > 64 is another kernel's job
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((256, 64), dtype=torch.bfloat16, device=DEV)
    D = torch.zeros((128, 256), device=DEV)
    assert _call(lib, 128, 256, 64, A, B, D, stream) == 3
    # more 128-column tiles of N than the array has counters for
    N = 16385 * 128
    A = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((N, 64), dtype=torch.bfloat16, device=DEV)
    D = torch.zeros((16, N), device=DEV)
    assert _call(lib, 16, N, 64, A, B, D, stream) == 3
    del B, D
    # more partial tiles than 16 MiB: M = 64, N = 38400, K = 4096 splits tiles in two
    A = torch.zeros((64, 4096), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((38400, 4096), dtype=torch.bfloat16, device=DEV)
    D = torch.zeros((64, 38400), device=DEV)
    plan = binding.gemm_query_plan(64, 38400, 4096, noalloc=True,
                                   sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan.kernel == 2
    assert plan.tiles * plan.splits * 128 * 64 * 4 > 16 << 20
    assert _call(lib, 64, 38400, 4096, A, B, D, stream) == 3
    assert binding.gemm_check_device_status() == binding.GEMM_OK
