"""Accumulating GEMM (D += alpha * A @ B.T through TMA reduce-add) vs the oracle.

The oracle of the accumulating form is the plain definition with C = D's
starting value and beta = 1: ref = alpha * sum_k a*b + D0, in fp64.  On
quarter-integer inputs every partial sum and every add is exact in float32,
so the result must match bit for bit whatever order the parts are added in.
Elsewhere the bound adds, to the accumulation bound 2e-3 * |alpha| * T, one
float32 rounding of the product and one of each add (parts + 1 of them).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_bits, device_status, run, to_f64
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_F32

pytestmark = pytest.mark.gpu

TILE_FORMS = [(1, 64), (1, 128), (1, 256), (3, 256), (4, 512), (5, 64), (5, 256), (6, 256),
              (7, 512), (8, 256), (9, 512), (10, 8)]
FORM_IDS = ["single64", "single128", "single256", "pair256", "pair512", "mcast64", "mcast256",
            "mcast8x256", "pairs2x512", "pairs2x256", "pairs4x512", "tiny"]


@pytest.fixture(autouse=True)
def _clean_status():
    binding.gemm_debug_inject(0)
    binding.gemm_set_wait_timeout(0)
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK
    yield
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK


def _problem(seed, M, N, K, dtype="bf16", values="quarter", alpha=0.5):
    """Random A, B and a starting D0 (drawn as the C of random_problem)."""
    p = workloads.random_problem(seed, M, N, K, dtype=dtype, values=values, with_c=True,
                                 alpha=alpha, beta=0.0)
    return workloads.Problem(f"acc_{M}x{N}x{K}", p.A, p.B, None, alpha=alpha, beta=0.0,
                             out=OUT_F32, D0=p.C, accumulate=True)


def _oracle(p, times=1):
    """D0 + times * alpha * A @ B.T (fp64) and T = sum |a||b|."""
    ref, absprod, _ = oracle.gemm(p.A, p.B, p.D0, times * p.alpha, 1.0)
    return ref, absprod


def _parts(p):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = binding.gemm_query_plan(p.M, p.N, p.K, sm_count=sms)
    return plan.splits if plan.kernel == 2 else 1


def _assert_close(D, p, ref, absprod, what, times=1):
    got = to_f64(D)
    a = abs(p.alpha) * times
    d0 = np.abs(p.D0.double().numpy())
    tol = 2e-3 * a * absprod + (_parts(p) * times + 1) * 2.0 ** -23 * (d0 + a * absprod) + 1e-5
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} outside; max err/tol {np.max(err / tol):.3g}"


@pytest.mark.parametrize("M,N,K", [(16, 300, 136), (48, 520, 4096), (64, 4096, 2048),
                                   (129, 257, 72), (300, 520, 264), (513, 700, 1000)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_accumulate_quarter_bit_exact(M, N, K, dtype):
    """The automatic choice: warp-level, tile and (for M <= 64 where it wins)
    skinny kernels."""
    for alpha in (0.5, -2.0):
        p = _problem(M + 3 * N + K, M, N, K, dtype=dtype, alpha=alpha)
        ref, _ = _oracle(p)
        assert_bits(run(p), ref, OUT_F32, f"{M}x{N}x{K} {dtype} alpha={alpha}")


@pytest.mark.parametrize("M,N,K", [(16, 300, 136), (48, 520, 4096), (64, 4096, 2048),
                                   (33, 130, 520)])
def test_accumulate_skinny_forced_bit_exact(M, N, K):
    """The skinny kernel on every M <= 64 shape (forced): each part of a split
    tile adds itself into D."""
    binding.gemm_debug_force_tile(2, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert binding.gemm_query_plan(M, N, K, sm_count=sms).kernel == 2
    p = _problem(M + 5 * N + K, M, N, K, dtype="bf16", alpha=0.5)
    ref, _ = _oracle(p)
    assert_bits(run(p), ref, OUT_F32, f"skinny {M}x{N}x{K}")


@pytest.mark.parametrize("form", TILE_FORMS, ids=FORM_IDS)
def test_every_tile_form_accumulate(form):
    binding.gemm_debug_force_tile(*form)
    p = _problem(61, 600, 400, 264)
    ref, _ = _oracle(p)
    assert_bits(run(p), ref, OUT_F32, f"accumulate form {form}")


def test_accumulate_twice_adds_twice():
    for M in (16, 300):
        p = _problem(62 + M, M, 384, 512)
        D = p.D0.to(DEV)
        A, B = p.A.to(DEV), p.B.to(DEV)
        binding.gemm_accumulate(A, B, D, alpha=p.alpha)
        binding.gemm_accumulate(A, B, D, alpha=p.alpha)
        ref, _ = _oracle(p, times=2)
        assert_bits(D, ref, OUT_F32, f"twice, M={M}")


@pytest.mark.parametrize("M,N,K", [(32, 2000, 4096), (1000, 520, 320)])
def test_accumulate_normal_within_tolerance(M, N, K):
    p = _problem(63, M, N, K, values="normal", alpha=0.75)
    ref, absprod = _oracle(p)
    _assert_close(run(p), p, ref, absprod, f"normal {M}x{N}x{K}")


def test_accumulate_tile_kernel_is_deterministic():
    """M > 64: one add per element, so repeated calls give identical bits."""
    p = _problem(64, 700, 600, 1024, values="normal")
    assert torch.equal(run(p), run(p))


@pytest.mark.parametrize("M", [20, 200])
def test_accumulate_unaligned_and_ragged_d(M):
    """Row pitch not a multiple of 16 bytes (atomic adds throughout), and N * 4 not
    a multiple of 16 (the chunk across column N by atomic adds)."""
    p = _problem(65 + M, M, 170, 96)
    ref, _ = _oracle(p)
    wide = torch.full((M, 171), 7.0, dtype=torch.float32, device=DEV)
    D = wide[:, :170]
    D.copy_(p.D0.to(DEV))
    run(p, D=D)
    assert_bits(D, ref, OUT_F32, "ldd = 171")
    assert torch.equal(wide[:, 170].cpu(), torch.full((M,), 7.0))
    wide = torch.full((M, 172), 7.0, dtype=torch.float32, device=DEV)
    D = wide[:, :170]  # ldd = 172: TMA boxes, the chunk across column N by atomic adds
    D.copy_(p.D0.to(DEV))
    run(p, D=D)
    assert_bits(D, ref, OUT_F32, "ldd = 172")
    assert torch.equal(wide[:, 170:].cpu(), torch.full((M, 2), 7.0))


def test_accumulate_k_zero_leaves_d():
    D = torch.randn(70, 90, device=DEV)
    before = D.clone()
    A = torch.empty((70, 0), dtype=torch.bfloat16, device=DEV)
    B = torch.empty((90, 0), dtype=torch.bfloat16, device=DEV)
    binding.gemm_accumulate(A, B, D, alpha=3.0)
    assert torch.equal(D, before)


def test_accumulate_skinny_workload_full():
    """16 x 28672 x 4096 with D starting as C: the MLP-shaped decode step."""
    p = workloads.skinny_accumulate_16x28672x4096()
    D = run(p)
    assert device_status() == binding.GEMM_OK
    ref, absprod = _oracle(p)
    _assert_close(D, p, ref, absprod, p.name)


def test_accumulate_mlp_sampled():
    """8192 x 28672 x 4096 with D starting as C; sampled entries."""
    A, B, C = workloads._mlp_draws(8192)
    D = C.to(DEV)
    binding.gemm_accumulate(A.to(DEV), B.to(DEV), D, alpha=0.5)
    assert device_status() == binding.GEMM_OK
    rng = np.random.default_rng(3)
    ii = np.concatenate([rng.integers(0, 8192, 4096), [0, 255, 256, 8191]])
    jj = np.concatenate([rng.integers(0, 28672, 4096), [0, 511, 512, 28671]])
    ref, absprod, _ = oracle.gemm_entries(A, B, ii, jj, C, 0.5, 1.0)
    got = to_f64(D[torch.from_numpy(ii).to(DEV), torch.from_numpy(jj).to(DEV)])
    d0 = np.abs(C.numpy()[ii, jj].astype(np.float64))
    tol = 1e-3 * absprod + 2 * 2.0 ** -23 * (d0 + 0.5 * absprod) + 1e-5
    assert (np.abs(got - ref) <= tol).all()
