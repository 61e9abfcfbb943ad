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
    if p.fp4:
        return binding.gemm_bf16_e2m1(A, B, p.Bs.to(DEV), C, D, alpha=p.alpha, beta=p.beta,
                                      out=p.out, stream=stream)
    if p.accumulate:
        if D is None:
            D = p.D0.to(DEV).contiguous()
        return binding.gemm_accumulate(A, B, D, alpha=p.alpha, stream=stream)
    if p.scatter:
        if D is None:
            D = (p.D0.to(DEV) if p.D0 is not None else
                 torch.zeros((p.d_rows, p.N), dtype=OUT_TORCH[p.out], device=DEV))
        return binding.gemm_scatter_rows(A, B, p.idx.to(DEV), D, C, alpha=p.alpha,
                                         beta=p.beta, stream=stream)
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


def oracle_scatter(p):
    """Expected D of a scattered problem: (ref, absprod, repeated, rows, row_abs, bad).

    ref / absprod are d_rows x N; rows no valid index names hold D0 (absprod
    0); rows named more than once are NaN and listed in `repeated` with the
    rows of the product that target them; `rows` / `row_abs` are the M rows
    the product sends (oracle values and sum |a||b|).
    """
    rows, absprod, bad = oracle.scatter_rows(p.A, p.B, p.idx, p.d_rows, p.C, p.alpha, p.beta)
    d0 = (p.D0.double().numpy() if p.D0 is not None else np.zeros((p.d_rows, p.N)))
    ref, repeated = oracle.scatter_place(d0, rows, p.idx.numpy())
    abs_d, _ = oracle.scatter_place(np.zeros_like(d0), absprod, p.idx.numpy())
    return ref, abs_d, repeated, rows, absprod, bad


def assert_scatter(D, p, exact, what=""):
    """Compare a scattered result with the oracle: rows named once (bits when
    `exact`, else the tolerance), rows named by no index unchanged bit for bit,
    and in rows named more than once each element equal to one sender's value."""
    ref, abs_d, repeated, rows, row_abs, _ = oracle_scatter(p)
    got = to_f64(D)
    idx = p.idx.numpy()
    named = np.zeros(p.d_rows, bool)
    valid = (idx >= 0) & (idx < p.d_rows)
    named[idx[valid]] = True
    once = named.copy()
    once[list(repeated)] = False
    if exact:
        assert_bits(D[torch.from_numpy(np.nonzero(once)[0]).to(D.device)],
                    ref[once], p.out, what + " (rows named once)")
    else:
        assert_within(got[once], ref[once], abs_d[once], p.out, what + " (rows named once)")
    d0 = p.D0.double().numpy() if p.D0 is not None else np.zeros((p.d_rows, p.N))
    same = (got[~named] == d0[~named]) | (np.isnan(got[~named]) & np.isnan(d0[~named]))
    assert same.all(), f"{what}: {(~same).sum()} elements of rows named by no index changed"
    for d, senders in repeated.items():
        cand = np.stack([expected_bits(rows[i][None, :], p.out)[0] for i in senders])
        if exact:
            ok = (cand == got[d][None, :]).any(axis=0)
        else:
            tol = tolerance(rows[senders], row_abs[senders], p.out)
            ok = (np.abs(cand - got[d][None, :]) <= tol).any(axis=0)
        assert ok.all(), f"{what}: row {d} (named by {senders}) holds a value none of them sent"


def device_status():
    return binding.gemm_check_device_status()
