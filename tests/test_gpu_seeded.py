"""Seeded GEMM (D = C + A @ B.T with C as the accumulator's start) vs the oracle.

The oracle is the plain definition with alpha = beta = 1.  On quarter-integer
inputs every running sum is exact in float32, so the seeded result matches bit
for bit.  Elsewhere the running sum, which holds C from the first K step on, is
rounded to float32 after each K step of 16: the bound adds ceil(K/16) ulps of
|C| + T to the usual accumulation bound.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_bits, device_status, to_f64
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F16, OUT_F32

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


def _seeded(p, D=None):
    return binding.gemm_seeded(p.A.to(DEV), p.B.to(DEV), p.C.to(DEV), D, out=p.out)


def _ref(p):
    ref, absprod, _ = oracle.gemm(p.A, p.B, p.C, 1.0, 1.0)
    return ref, absprod


@pytest.mark.parametrize("M,N,K", [(16, 8, 32), (64, 128, 128), (16, 300, 136), (48, 520, 600),
                                   (129, 257, 72), (300, 520, 264), (513, 700, 1000)])
@pytest.mark.parametrize("out", [OUT_F32, OUT_BF16, OUT_F16])
def test_seeded_quarter_bit_exact(M, N, K, out):
    """Warp-level kernel (tiny shapes), tile kernel (M <= 64 included)."""
    p = workloads.random_problem(M + 5 * N + K, M, N, K, dtype="bf16", values="quarter",
                                 with_c=True, out=out)
    ref, _ = _ref(p)
    assert_bits(_seeded(p), ref, out, f"seeded {M}x{N}x{K} out={out}")


@pytest.mark.parametrize("form", TILE_FORMS, ids=FORM_IDS)
def test_every_form_seeded(form):
    """Every tile form (pairs, multicast clusters, two-half accumulators) and the
    warp-level kernel; 4000 x 4000 gives every form more tiles than CTAs, so the
    epilogue also seeds the next tile of an accumulator while draining one."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.random_problem(71, 4000, 4000, 136, dtype="f16", values="quarter",
                                 with_c=True)
    ref, _ = _ref(p)
    assert_bits(_seeded(p), ref, OUT_F32, f"seeded form {form}")


def test_seeded_in_place():
    p = workloads.random_problem(72, 700, 600, 200, dtype="bf16", values="quarter", with_c=True)
    ref, _ = _ref(p)
    D = p.C.to(DEV)
    out = binding.gemm_seeded(p.A.to(DEV), p.B.to(DEV), D, D)
    assert out is D
    assert_bits(D, ref, OUT_F32, "in place")


def test_seeded_k_zero_is_c():
    C = torch.randn(300, 200)
    A = torch.empty((300, 0), dtype=torch.bfloat16, device=DEV)
    B = torch.empty((200, 0), dtype=torch.bfloat16, device=DEV)
    D = binding.gemm_seeded(A, B, C.to(DEV))
    assert torch.equal(D.cpu(), C)


@pytest.mark.parametrize("M,N,K", [(1000, 520, 320), (32, 2000, 2048)])
def test_seeded_normal_within_tolerance(M, N, K):
    p = workloads.random_problem(73, M, N, K, dtype="bf16", with_c=True)
    ref, absprod = _ref(p)
    got = to_f64(_seeded(p))
    steps = -(-K // 16)
    tol = 2e-3 * absprod + steps * 2.0 ** -23 * (np.abs(p.C.double().numpy()) + absprod) + 1e-5
    err = np.abs(got - ref)
    assert (err <= tol).all(), f"max err/tol {np.max(err / tol):.3g}"


@pytest.mark.parametrize("form", [(10, 8), (1, 64), (3, 256), (4, 512)],
                         ids=["tiny", "single64", "pair256", "pair512"])
def test_seed_enters_the_first_k_step(form):
    """C = 2^24 and two products of 1 in different K steps of 16.  Seeded, each
    step rounds 2^24 + 1 back to 2^24 (fp32 has no odd integers there), so
    D = 2^24; with C added once at the end the sum is 2 and D = 2^24 + 2."""
    binding.gemm_debug_force_tile(*form)
    M, N, K = 256, 256, 32
    a = np.zeros((M, K), np.float32)
    a[:, 0] = 1.0
    a[:, 16] = 1.0
    A = torch.from_numpy(a).to(torch.bfloat16).to(DEV)
    B = A[:N].clone()
    C = torch.full((M, N), 2.0 ** 24, device=DEV)
    seeded = binding.gemm_seeded(A, B, C)
    fused = binding.gemm_bf16(A, B, C, alpha=1.0, beta=1.0)
    assert torch.all(seeded == 2.0 ** 24), seeded.unique()
    assert torch.all(fused == 2.0 ** 24 + 2.0), fused.unique()


def test_seeded_equals_fused_on_exact_inputs():
    """Where every sum is exact, the order of adding C does not matter."""
    p = workloads.random_problem(74, 777, 640, 512, dtype="bf16", values="quarter",
                                 with_c=True)
    A, B, C = p.A.to(DEV), p.B.to(DEV), p.C.to(DEV)
    assert torch.equal(binding.gemm_seeded(A, B, C), binding.gemm_bf16(A, B, C))
