"""Shared pieces of the GPU parity tests: run a Problem through the C ABI and
compare with the oracle.

Tolerance (floating point): |D - ref| <= 2e-3 * T + 1e-5 with T = sum_k |a||b|,
the bound the build targets for float32 outputs.  For 16-bit outputs the final
round-to-nearest-even adds at most half an ulp of the output type, so the bound
grows by |ref| * 2^-8 (bf16) or |ref| * 2^-11 (f16).  Exact cases (quarter-
integer inputs) compare bits: float32(ref), then rounded to the output type.
"""
import numpy as np
import torch

import oracle
from tensor_core_gemm_02_gb300 import binding
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F16, OUT_F32, OUT_TORCH

DEV = "cuda"


def run(p, D=None, stream=None):
    """Launch the problem on the GPU through the library; returns D (device)."""
    A, B = p.A.to(DEV), p.B.to(DEV)
    C = p.C.to(DEV) if p.C is not None else None
    if p.idx is not None:
        return binding.gemm_gather_rows(A, p.idx.to(DEV), B, C, D, alpha=p.alpha,
                                        beta=p.beta, out=p.out, stream=stream)
    fn = binding.gemm_bf16 if A.dtype == torch.bfloat16 else binding.gemm_f16
    return fn(A, B, C, D, alpha=p.alpha, beta=p.beta, out=p.out, stream=stream)


def to_f64(D):
    return D.float().cpu().numpy().astype(np.float64)


def expected_bits(ref, out):
    """float32(ref) rounded to the output type, as float64 (exact cases)."""
    r32 = torch.from_numpy(ref.astype(np.float32))
    return r32.to(OUT_TORCH[out]).float().numpy().astype(np.float64)


def tolerance(ref, absprod, out):
    tol = 2e-3 * absprod + 1e-5
    if out == OUT_BF16:
        tol = tol + np.abs(ref) * 2.0 ** -8
    elif out == OUT_F16:
        tol = tol + np.abs(ref) * 2.0 ** -11
    return tol


def assert_within(D, ref, absprod, out, what=""):
    got = to_f64(D) if isinstance(D, torch.Tensor) else D
    err = np.abs(got - ref)
    tol = tolerance(ref, absprod, out)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {i.tolist()}; "
            f"max err/tol {np.max(err / np.maximum(tol, 1e-30)):.3g}")


def assert_bits(D, ref, out, what=""):
    got = to_f64(D)
    want = expected_bits(ref, out)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    if not same.all():
        i = np.argwhere(~same)[:5]
        raise AssertionError(f"{what}: {(~same).sum()} of {same.size} differ; first {i.tolist()}")


def oracle_full(p):
    return oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta, idx=p.idx)


def device_status():
    return binding.gemm_check_device_status()
