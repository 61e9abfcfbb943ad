"""Dependent GEMMs back to back, and concurrent streams (needs a GB300).

The kernels start their set-up while the previous kernel in the stream is still
running (programmatic dependent launch) and read their inputs only after it has
finished.  A chain where each GEMM consumes the previous one's output checks that
ordering.  Inputs in {-1, 0, 1} times signed selector matrices keep every intermediate
in {-1, 0, 1}, exact in bf16, so results compare bit for bit with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, device_status
from tensor_core_gemm_02_gb300 import binding
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F32

pytestmark = pytest.mark.gpu


def _ternary(rng, shape):
    return torch.from_numpy(rng.integers(-1, 2, shape).astype(np.float32)).to(torch.bfloat16)


def _signed_selector(rng, n, k):
    """n x k with one entry of +-1 per row: column j of A @ B^T is +-A[:, sel[j]],
    so values in {-1, 0, 1} stay there through any number of steps."""
    b = np.zeros((n, k), np.float32)
    b[np.arange(n), rng.integers(0, k, n)] = rng.choice([-1.0, 1.0], n)
    return torch.from_numpy(b).to(torch.bfloat16)


def _as_bf16(ref):
    assert np.array_equal(ref, np.round(ref)) and np.all(np.abs(ref) <= 256)
    return torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("M", [16, 48, 300, 1024])
def test_chain_of_dependent_gemms(M):
    """Eight GEMMs on one stream, each reading the previous one's bf16 output.
    M = 16 runs the warp-level kernel, larger M the tile kernels."""
    rng = np.random.default_rng(M)
    K = 192
    a = _ternary(rng, (M, K))
    bs = [_signed_selector(rng, K, K) for _ in range(8)]
    want = a
    for b in bs:
        want = _as_bf16(oracle.gemm(want, b)[0])
    x = a.to(DEV)
    for b in bs:
        x = binding.gemm_bf16(x, b.to(DEV), out=OUT_BF16)
    assert device_status() == binding.GEMM_OK
    assert torch.equal(x.cpu(), want)


def test_chain_mixing_kernels():
    """Warp-level -> gathered tile -> skinny on one stream, each step reading the
    previous one's output."""
    rng = np.random.default_rng(5)
    a = _ternary(rng, (16, 128))
    b1 = _signed_selector(rng, 256, 128)
    idx = torch.from_numpy(rng.integers(0, 16, 512).astype(np.int32))
    b2 = _signed_selector(rng, 640, 256)
    b3 = _signed_selector(rng, 64, 640)  # K >= 8 N: the skinny kernel for 40 rows

    d1 = binding.gemm_bf16(a.to(DEV), b1.to(DEV), out=OUT_BF16)           # 16 x 256
    d2 = binding.gemm_gather_rows(d1, idx.to(DEV), b2.to(DEV), out=OUT_BF16)  # 512 x 640
    d3 = binding.gemm_bf16(d2[:40], b3.to(DEV), out=OUT_F32)              # 40 x 64
    assert device_status() == binding.GEMM_OK

    r1 = _as_bf16(oracle.gemm(a, b1)[0])
    r2 = _as_bf16(oracle.gemm(r1, b2, idx=idx)[0])
    r3 = oracle.gemm(r2[:40].contiguous(), b3)[0]
    assert np.array_equal(d3.cpu().numpy().astype(np.float64), r3)


def test_concurrent_streams_skinny_and_tile():
    """Skinny GEMMs on two streams at once (each stream has its own scratch) and a
    tile GEMM on a third; every result checked."""
    rng = np.random.default_rng(9)
    K, N = 1024, 8192
    problems = []
    for _ in range(2):
        a = _ternary(rng, (16, K))
        b = _ternary(rng, (N, K))
        problems.append((a, b))
    big_a, big_b = _ternary(rng, (1024, K)), _ternary(rng, (2048, K))
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = []
    for rep in range(3):
        for (a, b), st in zip(problems, streams[:2]):
            with torch.cuda.stream(st):
                outs.append((a, b, binding.gemm_bf16(a.to(DEV), b.to(DEV), stream=st)))
        with torch.cuda.stream(streams[2]):
            outs.append((big_a, big_b,
                         binding.gemm_bf16(big_a.to(DEV), big_b.to(DEV), stream=streams[2])))
    torch.cuda.synchronize()
    assert device_status() == binding.GEMM_OK
    for a, b, d in outs:
        ref, _, _ = oracle.gemm(a, b)
        assert np.array_equal(d.cpu().numpy().astype(np.float64), ref)
