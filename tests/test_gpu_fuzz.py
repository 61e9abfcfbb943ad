"""Seeded random sweep over shapes, kernel forms, entry points and output types
(needs a GB300).

Every case uses quarter-integer inputs (and scales near 1 for FP4 weights), so
every partial sum is exact in float32 and each result is compared bit for bit
with the oracle, whatever kernel or summation order ran.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_bits, assert_scatter, device_status, run
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F16, OUT_F32

pytestmark = pytest.mark.gpu

FORMS = [(0, 0), (1, 64), (1, 128), (1, 256), (3, 256), (4, 512), (5, 64), (5, 256), (6, 256),
         (7, 512), (8, 256), (9, 512), (10, 8)]
KINDS = ["plain", "gather", "scatter", "accumulate", "seeded", "fp4"]


def _case(i):
    rng = np.random.default_rng(1000 + i)
    kind = KINDS[i % len(KINDS)]
    M = int(rng.choice([1, 7, 16, 40, 64, 65, 130, 300, 513]))
    N = int(rng.choice([8, 33, 100, 256, 300, 520, 1000]))
    K = int(rng.choice([0, 16, 32, 72, 136, 264, 520, 1024])) if kind != "fp4" else \
        int(rng.choice([32, 64, 96, 256, 512, 1024]))
    form = FORMS[int(rng.integers(0, len(FORMS)))]
    dtype = "bf16" if kind == "fp4" else str(rng.choice(["bf16", "f16"]))
    out = OUT_F32 if kind in ("accumulate", "seeded", "fp4") and rng.random() < 0.5 else \
        int(rng.choice([OUT_F32, OUT_BF16, OUT_F16]))
    if kind == "accumulate":
        out = OUT_F32
    return kind, M, N, K, form, dtype, out, int(rng.integers(0, 2**31))


@pytest.mark.parametrize("i", range(60))
def test_fuzz_bit_exact(i):
    kind, M, N, K, form, dtype, out, seed = _case(i)
    what = f"{kind} {M}x{N}x{K} form={form} {dtype} out={out}"
    binding.gemm_debug_force_tile(*form)
    try:
        if kind == "plain":
            p = workloads.random_problem(seed, M, N, K, dtype=dtype, values="quarter",
                                         with_c=seed % 2 == 0, alpha=0.5, beta=-1.0, out=out)
            ref, _, _ = oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta)
            assert_bits(run(p), ref, out, what)
        elif kind == "gather":
            p = workloads.random_problem(seed, M, N, K, dtype=dtype, values="quarter",
                                         with_c=True, alpha=2.0, beta=0.5, out=out,
                                         gather_rows=max(1, M // 2 + 3))
            ref, _, _ = oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta, idx=p.idx)
            assert_bits(run(p), ref, out, what)
        elif kind == "scatter":
            p = workloads.random_problem(seed, M, N, K, dtype=dtype, values="quarter",
                                         with_c=True, alpha=0.5, beta=2.0, out=out,
                                         scatter_rows=M + 37, repeats=seed % 3 == 0)
            assert_scatter(run(p), p, True, what)
        elif kind == "accumulate":
            q = workloads.random_problem(seed, M, N, K, dtype=dtype, values="quarter",
                                         with_c=True, alpha=-0.5)
            p = workloads.Problem("acc", q.A, q.B, None, alpha=q.alpha, beta=0.0, out=OUT_F32,
                                  D0=q.C, accumulate=True)
            ref, _, _ = oracle.gemm(q.A, q.B, q.C, q.alpha, 1.0)
            assert_bits(run(p), ref, OUT_F32, what)
        elif kind == "seeded":
            p = workloads.random_problem(seed, M, N, K, dtype=dtype, values="quarter",
                                         with_c=True, out=out)
            ref, _, _ = oracle.gemm(p.A, p.B, p.C, 1.0, 1.0)
            D = binding.gemm_seeded(p.A.to(DEV), p.B.to(DEV), p.C.to(DEV), out=out)
            assert_bits(D, ref, out, what)
        else:  # fp4 weights, scales 2^-2 .. 2^2
            rng = np.random.default_rng(seed)
            A = torch.from_numpy((rng.integers(-4, 5, (M, K)) / 4).astype(np.float32)).to(
                torch.bfloat16)
            Bq = torch.from_numpy(rng.integers(0, 256, (N, K // 2)).astype(np.uint8))
            Bs = torch.from_numpy(rng.integers(125, 130, (K // 32, N)).astype(np.uint8))
            C = torch.from_numpy((rng.integers(-4, 5, (M, N)) / 4).astype(np.float32))
            ref, _ = oracle.w4(A, Bq.numpy(), Bs.numpy(), C, 0.5, 1.0)
            D = binding.gemm_bf16_e2m1(A.to(DEV), Bq.to(DEV), Bs.to(DEV), C.to(DEV), alpha=0.5,
                                       beta=1.0, out=out)
            assert_bits(D, ref, out, what)
    finally:
        binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK, what
