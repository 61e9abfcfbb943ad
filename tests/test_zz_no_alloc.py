"""The allocation-free skinny entry point (gemm_skinny_noalloc) on the GPU.

This entry point is for callers that cannot call cudaMalloc where they run the
GEMM (their device memory belongs to another allocator, or they are in a
section where cudaMalloc's implicit synchronisation is not allowed).  It keeps
its scratch in a fixed array inside the library instead.  Here it is called
through the C ABI and its output is compared with the oracle, element by
element, on two calls in a row (the second call finds the array as the first
one left it): bit for bit on quarter-integer inputs (every partial sum is exact
in float32, whatever order the K sum takes), within the parity tolerance on
normal inputs.  Around the second call neither the free device memory nor
PyTorch's allocated bytes may change.

The file name makes pytest collect it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_bits, assert_within
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F16, OUT_F32, OUT_TORCH

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(lib, p, A, B, C, D, stream):
    return lib.gemm_skinny_noalloc(
        p.M, p.N, p.K, 1 if p.A.dtype == torch.bfloat16 else 0, A.data_ptr(), A.stride(0),
        B.data_ptr(), B.stride(0), C.data_ptr() if C is not None else None,
        C.stride(0) if C is not None else 0, D.data_ptr(), D.stride(0), p.out,
        ctypes.c_float(p.alpha), ctypes.c_float(p.beta), ctypes.c_void_p(stream))


def _twice(p, check):
    """Two calls in a row into a NaN-filled D, each checked; the second call is
    also checked to allocate no device memory."""
    A, B = p.A.to(DEV), p.B.to(DEV)
    C = p.C.to(DEV) if p.C is not None else None
    D = torch.empty((p.M, p.N), dtype=OUT_TORCH[p.out], device=DEV)
    lib = binding.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        D.fill_(float("nan"))
        torch.cuda.synchronize()
        free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        st = _noalloc(lib, p, A, B, C, D, stream)
        assert st == binding.GEMM_OK, binding.gemm_status_string(st)
        assert binding.gemm_check_device_status() == binding.GEMM_OK
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free0, "the call allocated device memory"
            assert torch.cuda.memory_allocated() == allocated0
        assert not torch.isnan(D.float()).any(), f"call {call}: elements not written"
        check(D, call)


# (M, N, K): 1, 16, 33, 48 and 64 rows.  For 17..64 rows with K < N (8192 x 4096)
# gemm_bf16 itself runs the tile kernel, while this entry point always runs the
# skinny one (64 rows: its eight-warp epilogue); 16 x 8 x 32 is small enough for
# the warp-level kernel.
SHAPES = [(1, 4096, 4096), (16, 28672, 4096), (33, 8192, 4096), (48, 2048, 8192),
          (64, 8192, 4096), (64, 640, 136), (16, 8, 32)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_noalloc_quarter_integers_match_oracle_twice(M, N, K, dtype):
    for out, with_c, alpha, beta in [(OUT_F32, True, 0.5, 1.0), (OUT_BF16, False, 2.0, 0.0),
                                     (OUT_F16, True, -1.0, 0.5)]:
        p = workloads.random_problem(M * 5 + N + K + out, M, N, K, dtype=dtype, values="quarter",
                                     with_c=with_c, alpha=alpha, beta=beta, out=out)
        ref, _, _ = oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta)
        _twice(p, lambda D, call: assert_bits(D, ref, out, f"{M}x{N}x{K} {dtype} out={out} "
                                                           f"call {call}"))


def test_noalloc_normal_inputs_within_tolerance_twice():
    """The decode shape with N(0,1) activations and N(0,0.02) weights, C, alpha = 0.5."""
    p = workloads.random_problem(41, 16, 28672, 4096, dtype="bf16", with_c=True, alpha=0.5,
                                 beta=1.0, b_scale=0.02)
    ref, absprod, _ = oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta)
    _twice(p, lambda D, call: assert_within(D, ref, absprod, OUT_F32, f"call {call}"))


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
