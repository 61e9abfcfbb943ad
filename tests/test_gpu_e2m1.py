"""Both operands FP4 (gemm_e2m1) on the GPU against the oracle (needs a GB300).

Exact inputs (codes of magnitude <= 2, scales 2^-1 .. 2^1, K <= 2^16) make
every product a multiple of 2^-4 below 16 and every partial sum exact in
float32, whatever order the tensor cores add them in: those results compare
bit for bit (16-bit outputs: the float32 value rounded once).  Random codes
and scales compare within the parity tolerance.  Every kernel form runs:
packed codes (MMA kind::mxf4) and the 16U4_ALIGN16B image (kind::mxf8f6f4),
single CTAs with tiles 128 and 256 wide, CTA pairs with 256 x 256 tiles, and the
swap-AB stream-K skinny form for M <= 64 (packed codes).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_bits, assert_within, device_status, to_f64
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F16, OUT_F32

pytestmark = pytest.mark.gpu

FORMS = [(11, 256), (11, 128), (12, 256), (12, 128), (13, 256), (14, 256)]
FORM_IDS = ["packed256", "packed128", "align16b256", "align16b128", "packed_pair", "align16b_pair"]


@pytest.fixture(autouse=True)
def _clean_status():
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK
    yield
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK


def run_e2m1(p, D=None):
    C = p.C.to(DEV) if p.C is not None else None
    return binding.gemm_e2m1(p.A.to(DEV), p.As.to(DEV), p.B.to(DEV), p.Bs.to(DEV), C, D,
                             alpha=p.alpha, beta=p.beta, out=p.out, image=p.image)


def oracle_e2m1(p, rows=None):
    return oracle.e2m1(p.A, p.As, p.B, p.Bs, p.C, p.alpha, p.beta, rows=rows)


CASES = [(OUT_F32, True, 0.5, 2.0), (OUT_BF16, False, 2.0, 0.0), (OUT_F16, True, -1.0, 0.5)]


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("M,N,K", [(129, 257, 256), (300, 520, 512), (256, 384, 1024),
                                   (1000, 96, 128), (16, 8, 128), (128, 256, 2048)])
def test_exact_every_form_bit_exact(form, M, N, K):
    """Ragged shapes over several tiles, K over several stages and partial ones."""
    binding.gemm_debug_force_tile(*form)
    image = 0 if form[0] in (11, 13) else 1
    for out, with_c, alpha, beta in CASES:
        p = workloads.e2m1_problem(M + 3 * N + K + out, M, N, K, values="exact", with_c=with_c,
                                   alpha=alpha, beta=beta, out=out, image=image)
        ref, _ = oracle_e2m1(p)
        assert_bits(run_e2m1(p), ref, out, f"form {form} {M}x{N}x{K} out={out}")


@pytest.mark.parametrize("form", [FORMS[0], FORMS[1], FORMS[4]], ids=[FORM_IDS[0], FORM_IDS[1], FORM_IDS[4]])
@pytest.mark.parametrize("K", [32, 96, 160, 288])
def test_packed_k_not_a_multiple_of_128(form, K):
    """Packed codes take any whole number of 32-element blocks: the last stage's
    codes and scale rows past K are zero fill (a zero code contributes nothing)."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.e2m1_problem(K, 200, 300, K, values="exact", with_c=True, alpha=0.5)
    ref, _ = oracle_e2m1(p)
    assert_bits(run_e2m1(p), ref, OUT_F32, f"form {form} K={K}")


@pytest.mark.parametrize("M,N,K", [(1, 300, 4096), (16, 8, 32), (16, 28672, 1024), (17, 640, 96),
                                   (33, 1000, 2048), (48, 256, 512), (64, 4096, 4096),
                                   (64, 130, 8192)])
def test_skinny_every_shape_bit_exact(M, N, K):
    """The swap-AB stream-K skinny form (M <= 64, packed codes): partial tiles of
    B, K split over CTAs, padded rows of A, every output type."""
    binding.gemm_debug_force_tile(15, 128)
    plan = binding.gemm_query_plan(M, N, K, e2m1=0, sm_count=148)
    assert plan.kernel == 15
    for out, with_c, alpha, beta in CASES:
        p = workloads.e2m1_problem(M * 11 + N + K + out, M, N, K, values="exact",
                                   with_c=with_c, alpha=alpha, beta=beta, out=out)
        ref, _ = oracle_e2m1(p)
        assert_bits(run_e2m1(p), ref, out, f"skinny {M}x{N}x{K} out={out}")


def test_skinny_random_within_tolerance_and_timeout():
    binding.gemm_debug_force_tile(15, 128)
    p = workloads.e2m1_problem(91, 40, 3000, 4096, with_c=True, alpha=0.5, beta=1.0)
    ref, absprod = oracle_e2m1(p)
    assert_within(run_e2m1(p), ref, absprod, OUT_F32, "skinny random")
    binding.gemm_set_wait_timeout(50_000_000)
    binding.gemm_debug_inject(1)
    try:
        run_e2m1(p)
        assert device_status() == binding.GEMM_ERR_TIMEOUT
    finally:
        binding.gemm_debug_inject(0)
        binding.gemm_set_wait_timeout(0)
    assert_within(run_e2m1(p), ref, absprod, OUT_F32, "skinny after timeout")


@pytest.mark.parametrize("image", [0, 1])
def test_decode_shape_full_exact(image):
    """16 x 28672 x 4096 (the decode shape), exact inputs, every element bit for bit."""
    p = workloads.e2m1_problem(70 + image, 16, 28672, 4096, values="exact", with_c=True,
                               alpha=0.5, image=image)
    ref, _ = oracle_e2m1(p)
    assert_bits(run_e2m1(p), ref, OUT_F32, f"decode shape image={image}")


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
def test_timeout_reports_and_recovers(form):
    """A stage that never completes (the test hook adds bytes to its expected
    count): the wait runs out, the status says so, nothing hangs, and the next
    call is exact."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.e2m1_problem(21, 512, 512, 512, values="exact",
                               image=0 if form[0] in (11, 13) else 1)
    binding.gemm_set_wait_timeout(50_000_000)
    binding.gemm_debug_inject(1)
    try:
        run_e2m1(p)
        assert device_status() == binding.GEMM_ERR_TIMEOUT
    finally:
        binding.gemm_debug_inject(0)
        binding.gemm_set_wait_timeout(0)
    ref, _ = oracle_e2m1(p)
    assert_bits(run_e2m1(p), ref, OUT_F32, "after timeout")


@pytest.mark.parametrize("image", [0, 1])
def test_1024_cubed_full_exact(image):
    """A multiple of 128 rows: 1024^3, exact inputs, bf16 out, every element."""
    p = workloads.e2m1_problem(80 + image, 1024, 1024, 1024, values="exact", out=OUT_BF16,
                               alpha=1.0, beta=0.0, image=image)
    ref, _ = oracle_e2m1(p)
    assert_bits(run_e2m1(p), ref, OUT_BF16, f"1024^3 image={image}")


@pytest.mark.parametrize("form", FORMS, ids=FORM_IDS)
def test_random_within_tolerance(form):
    """Every code and scales of the workloads' ranges: within the parity tolerance."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.e2m1_problem(90, 384, 1000, 2048, with_c=True, alpha=0.5, beta=1.0,
                               image=0 if form[0] in (11, 13) else 1)
    ref, absprod = oracle_e2m1(p)
    assert_within(run_e2m1(p), ref, absprod, OUT_F32, f"form {form}")


def test_decode_workload_full():
    """The e2m1_16x28672x4096 workload (random codes), every element."""
    p = workloads.e2m1_16x28672x4096()
    ref, absprod = oracle_e2m1(p)
    assert_within(run_e2m1(p), ref, absprod, p.out, p.name)


def test_8192_workload_sampled_rows():
    """The e2m1_8192 workload (the size the bench times): 48 whole rows -- the
    first, last and a middle block's worth -- against the oracle."""
    p = workloads.e2m1_8192()
    D = run_e2m1(p)
    torch.cuda.synchronize()
    for r0 in (0, 4096 + 64, 8192 - 16):
        ref, absprod = oracle_e2m1(p, rows=(r0, r0 + 16))
        assert_within(D[r0:r0 + 16], ref, absprod, p.out, f"{p.name} rows {r0}..{r0 + 16}")


def test_both_images_agree_on_exact_inputs():
    """The packed and the 16U4 forms take the same products: equal bit for bit
    where every partial sum is exact."""
    p = workloads.e2m1_problem(5, 512, 768, 1024, values="exact", with_c=True, alpha=0.5)
    d0 = run_e2m1(p)
    p.image = 1
    d1 = run_e2m1(p)
    assert torch.equal(d0, d1)


def test_k_zero_and_in_place():
    """K = 0 gives beta * C; C == D (float32, same pitch) is an exact in-place update."""
    M, N = 200, 300
    rng = np.random.default_rng(3)
    C = torch.from_numpy((rng.integers(-4, 5, (M, N)) / 4).astype(np.float32)).to(DEV)
    empty_q = torch.empty((M, 0), dtype=torch.uint8, device=DEV)
    empty_bq = torch.empty((N, 0), dtype=torch.uint8, device=DEV)
    D = binding.gemm_e2m1(empty_q, torch.empty((0, M), dtype=torch.uint8, device=DEV), empty_bq,
                          torch.empty((0, N), dtype=torch.uint8, device=DEV), C, alpha=3.0,
                          beta=0.5)
    assert torch.equal(D, 0.5 * C)
    p = workloads.e2m1_problem(9, M, N, 256, values="exact", with_c=True, alpha=0.5)
    ref, _ = oracle_e2m1(p)
    Cd = p.C.to(DEV)
    binding.gemm_e2m1(p.A.to(DEV), p.As.to(DEV), p.B.to(DEV), p.Bs.to(DEV), Cd, Cd, alpha=0.5,
                      beta=1.0)
    assert_bits(Cd, ref, OUT_F32, "in place")


def test_unaligned_scales_are_copied():
    """Scale rows with a pitch that is not a multiple of 16 bytes (M = 200, N = 300
    given as slices of wider buffers at odd offsets) go through the library's
    padded copy and give the same bits."""
    p = workloads.e2m1_problem(11, 200, 300, 512, values="exact", with_c=True, alpha=0.5)
    ref, _ = oracle_e2m1(p)
    big_a = torch.zeros((p.K // 32, 203), dtype=torch.uint8, device=DEV)
    big_b = torch.zeros((p.K // 32, 305), dtype=torch.uint8, device=DEV)
    As = big_a[:, 1:201]
    Bs = big_b[:, 3:303]
    As.copy_(p.As.to(DEV))
    Bs.copy_(p.Bs.to(DEV))
    D = binding.gemm_e2m1(p.A.to(DEV), As, p.B.to(DEV), Bs, p.C.to(DEV), alpha=0.5, beta=1.0)
    assert_bits(D, ref, OUT_F32, "unaligned scales")


def test_nan_scale_gives_nan():
    """A scale byte of 255 stands for NaN: the rows (of D) whose A block carries it
    are NaN, others are exact."""
    p = workloads.e2m1_problem(12, 128, 256, 256, values="exact", alpha=1.0, beta=0.0)
    p.As[3, 5] = 255   # block 3 of row 5 of A
    ref, _ = oracle_e2m1(p)
    got = to_f64(run_e2m1(p))
    assert np.isnan(got[5]).all() and np.isnan(ref[5]).all()
    keep = np.ones(128, bool)
    keep[5] = False
    assert np.array_equal(got[keep], ref[keep].astype(np.float32).astype(np.float64))


def test_skinny_nan_scale_gives_nan():
    """The skinny form (16 rows, K split over CTAs): a NaN scale byte of A makes
    its row of D NaN through the split tiles' partial sums; the other rows are
    exact."""
    p = workloads.e2m1_problem(14, 16, 2000, 4096, values="exact", alpha=1.0, beta=0.0)
    assert binding.gemm_query_plan(16, 2000, 4096, e2m1=0).kernel == 15
    p.As[40, 5] = 255   # block 40 of row 5 of A
    ref, _ = oracle_e2m1(p)
    got = to_f64(run_e2m1(p))
    assert np.isnan(got[5]).all() and np.isnan(ref[5]).all()
    keep = np.ones(16, bool)
    keep[5] = False
    assert np.array_equal(got[keep], ref[keep].astype(np.float32).astype(np.float64))
