"""GPU path vs the oracle, element by element (needs a GB300)."""
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (DEV, assert_bits, assert_within, device_status, expected_bits, oracle_full,
                         run, to_f64)
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F16, OUT_F32

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(autouse=True)
def _clean_status():
    binding.gemm_debug_inject(0)
    binding.gemm_set_wait_timeout(0)
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK
    yield
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK


TILE_FORMS = [(1, 64), (1, 128), (1, 256), (3, 256), (4, 512), (5, 64), (5, 256), (6, 256),
              (7, 512), (8, 256), (9, 512), (10, 8)]
FORM_IDS = ["single64", "single128", "single256", "pair256", "pair512", "mcast64", "mcast256",
            "mcast8x256", "pairs2x512", "pairs2x256", "pairs4x512", "tiny"]


@pytest.mark.parametrize("form", TILE_FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("M,N,K", [(129, 257, 72), (300, 520, 264), (513, 700, 1000),
                                   (256, 256, 64), (1000, 96, 136)])
def test_every_tile_form_bit_exact(form, M, N, K):
    """Each tile kernel form, forced, on ragged multi-tile shapes with exact inputs."""
    binding.gemm_debug_force_tile(*form)
    for dtype, out, with_c, alpha, beta in [("bf16", OUT_F32, True, 0.5, 2.0),
                                            ("f16", OUT_BF16, False, 1.0, 0.0),
                                            ("bf16", OUT_F16, True, -1.0, 1.0)]:
        p = workloads.random_problem(M + 3 * N + K, M, N, K, dtype=dtype, values="quarter",
                                     with_c=with_c, alpha=alpha, beta=beta, out=out)
        ref, _, _ = oracle_full(p)
        assert_bits(run(p), ref, out, f"form {form} {M}x{N}x{K} {dtype} out={out}")


@pytest.mark.parametrize("form", TILE_FORMS, ids=FORM_IDS)
def test_every_tile_form_gather(form):
    binding.gemm_debug_force_tile(*form)
    p = workloads.random_problem(42, 600, 400, 264, dtype="bf16", values="quarter",
                                 with_c=True, alpha=0.5, gather_rows=333)
    ref, _, _ = oracle_full(p)
    assert_bits(run(p), ref, OUT_F32, f"gather form {form}")


@pytest.mark.parametrize("form", TILE_FORMS[:-1], ids=FORM_IDS[:-1])  # (the tiny kernel has no waits)
def test_every_tile_form_timeout(form):
    binding.gemm_debug_force_tile(*form)
    p = workloads.random_problem(43, 512, 512, 256, dtype="bf16", values="quarter")
    binding.gemm_set_wait_timeout(50_000_000)
    binding.gemm_debug_inject(1)
    try:
        run(p)
        assert device_status() == binding.GEMM_ERR_TIMEOUT
    finally:
        binding.gemm_debug_inject(0)
        binding.gemm_set_wait_timeout(0)
    ref, _, _ = oracle_full(p)
    assert_bits(run(p), ref, OUT_F32, f"after timeout, form {form}")


def test_worked_example_bit_exact():
    """The mma.sync page's 16 x 8 x 32 example: D equals the stored exact result."""
    p = workloads.worked_16x8x32()
    D = run(p)
    stored = np.loadtxt(os.path.join(GOLDEN, "worked_16x8x32.txt"))
    assert np.array_equal(to_f64(D), stored)


@pytest.mark.parametrize("form", TILE_FORMS + [(2, 128)], ids=FORM_IDS + ["skinny"])
def test_worked_example_every_form(form):
    """The same 16 x 8 x 32 inputs through every kernel form, forced: a 16 x 8
    corner of a 128- or 256-row tile, so the TMA boxes of A (128 x 64 or more)
    and B read mostly out-of-bounds zero fill (K = 32 of a 64-wide block, 8 of
    up to 512 columns; the second CTA of a pair and all but one CTA of a
    cluster load boxes that lie wholly outside), and D's stores are clipped to
    8 columns and 16 rows.  D must equal the stored exact result bit for bit."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.worked_16x8x32()
    plan = binding.gemm_query_plan(p.M, p.N, p.K, sm_count=148)
    assert plan.kernel == form[0]
    D = run(p)
    stored = np.loadtxt(os.path.join(GOLDEN, "worked_16x8x32.txt"))
    assert np.array_equal(to_f64(D), stored), f"form {form}"


QUARTER_SHAPES = [(1, 1, 8), (16, 8, 32), (5, 3, 24), (127, 255, 64), (128, 256, 64),
                  (129, 257, 72), (300, 520, 264), (257, 129, 520), (64, 640, 136),
                  (384, 96, 1000)]


@pytest.mark.parametrize("M,N,K", QUARTER_SHAPES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_quarter_integers_bit_exact(M, N, K, dtype):
    """Quarter-integer inputs make every partial sum exact: D must match bit for bit."""
    for out, with_c, alpha, beta in [(OUT_F32, False, 1.0, 1.0), (OUT_F32, True, 0.5, 2.0),
                                     (OUT_BF16, True, -1.0, 0.5), (OUT_F16, False, 2.0, 0.0)]:
        p = workloads.random_problem(M * 7 + N + K, M, N, K, dtype=dtype, values="quarter",
                                     with_c=with_c, alpha=alpha, beta=beta, out=out)
        ref, _, _ = oracle_full(p)
        assert_bits(run(p), ref, out, f"{M}x{N}x{K} {dtype} out={out} C={with_c}")


def test_fma_single_rounding():
    """alpha*acc + C must be one fused rounding (fma page): 2^-11 + 2^-24, not 2^-11."""
    K = 8
    a = torch.zeros((1, K), dtype=torch.float16)
    a[0, 0], a[0, 1] = 1.0, 2.0 ** -12
    b = torch.zeros((1, K), dtype=torch.float16)
    b[0, 0], b[0, 1] = 1.0, 1.0
    c = torch.full((1, 1), -1.0)
    alpha = float(np.float32(1 + 2.0 ** -12))
    D = binding.gemm_f16(a.to(DEV), b.to(DEV), c.to(DEV), alpha=alpha, beta=1.0)
    assert D.item() == 2.0 ** -11 + 2.0 ** -24


def test_two_a_plus_one():
    """The fma page's example through the GEMM: X * I^T * 2 + 1 == 2X + 1 exactly."""
    rng = np.random.default_rng(7)
    K = 64
    X = torch.from_numpy(rng.integers(-64, 65, (40, K)).astype(np.float16))
    eye = torch.eye(K, dtype=torch.float16)
    ones = torch.ones((40, K))
    D = binding.gemm_f16(X.to(DEV), eye.to(DEV), ones.to(DEV), alpha=2.0, beta=1.0)
    assert torch.equal(D.cpu(), 2 * X.float() + 1)


NORMAL_SHAPES = [(777, 1000, 520), (128, 4096, 64), (1000, 333, 1032), (2, 5000, 256)]


@pytest.mark.parametrize("M,N,K", NORMAL_SHAPES)
@pytest.mark.parametrize("out", [OUT_F32, OUT_BF16, OUT_F16])
def test_normal_within_tolerance(M, N, K, out):
    p = workloads.random_problem(M + N + K + out, M, N, K, dtype="bf16", with_c=True,
                                 alpha=0.5, beta=1.0, out=out, b_scale=0.02)
    ref, absprod, _ = oracle_full(p)
    assert_within(run(p), ref, absprod, out, f"{M}x{N}x{K}")


def test_f16_1024_full():
    """f16 1024^3 with C (alpha = beta = 1), every element."""
    p = workloads.f16_1024()
    ref, absprod, _ = oracle_full(p)
    assert_within(run(p), ref, absprod, p.out, p.name)


def _full_check(p, rows_per_chunk=512):
    """Every element of D against the oracle, a block of rows at a time (the
    oracle's float64 result for the whole matrix would not need to be held)."""
    D = run(p)
    torch.cuda.synchronize()
    got_all = D.cpu()
    del D
    for i0 in range(0, p.M, rows_per_chunk):
        i1 = min(p.M, i0 + rows_per_chunk)
        ref, absprod, bad = oracle.gemm(p.A, p.B, p.C, p.alpha, p.beta, idx=p.idx,
                                        rows=(i0, i1))
        assert not bad
        assert_within(to_f64(got_all[i0:i1]), ref, absprod, p.out, f"{p.name} rows {i0}..{i1}")


def test_bf16_8192_full():
    """bf16 8192^3, bf16 out: all 67,108,864 elements."""
    _full_check(workloads.bf16_8192())


def test_mlp_full():
    """8192 x 28672 x 4096 with D = fma(0.5, A B^T, 1.0 C): all 234,881,024 elements."""
    _full_check(workloads.mlp_8192x28672x4096(), rows_per_chunk=256)


def test_skinny_full():
    p = workloads.skinny_16x28672x4096()
    ref, absprod, _ = oracle_full(p)
    assert_within(run(p), ref, absprod, p.out, p.name)


def test_gather_full():
    """16384 rows gathered from a 65536-row table, N = K = 4096: all 67,108,864 elements."""
    _full_check(workloads.gather_16384_of_65536())


@pytest.mark.parametrize("out,with_c", [(OUT_F32, True), (OUT_BF16, False)])
def test_gather_split_into_waves_and_tail_exact(out, with_c):
    """16484 gathered rows, N = 4096, K = 2048: the clustered form (four CTA pairs
    sharing rows) runs the first 15360 rows as whole waves and single CTAs on the
    SMs it leaves idle run the other 1124 (a ragged last stripe).  Quarter-integer
    inputs make every sum exact, so sampled entries -- around the boundary, in the
    tail, anywhere -- match the oracle bit for bit (bf16 output: the oracle's value
    rounded once), as does the same call with the clustered form forced for all
    rows."""
    p = workloads.random_problem(31, 16484, 4096, 2048, dtype="bf16", values="quarter",
                                 with_c=with_c, alpha=0.5, beta=-1.0, gather_rows=4096,
                                 out=out)
    D = run(p)
    rng = np.random.default_rng(7)
    ii = np.concatenate([rng.integers(0, p.M, 2048), rng.integers(15360 - 256, 15360 + 256, 1024),
                         rng.integers(15360, p.M, 1024), np.array([15359, 15360, p.M - 1])])
    jj = np.concatenate([rng.integers(0, p.N, 4096), np.array([0, p.N - 1, 2047])])
    ref, _, _ = oracle.gemm_entries(p.A, p.B, ii, jj, p.C, p.alpha, p.beta, idx=p.idx)
    got = D[torch.from_numpy(ii).to(DEV), torch.from_numpy(jj).to(DEV)]
    assert np.array_equal(to_f64(got), expected_bits(ref, out))
    binding.gemm_debug_force_tile(9, 512)
    try:
        forced = run(p)
    finally:
        binding.gemm_debug_force_tile(0, 0)
    assert torch.equal(D, forced)
    assert device_status() == binding.GEMM_OK


@pytest.mark.parametrize("form", [(1, 128), (4, 512)], ids=["two_issuers", "pair512"])
def test_gather_identity_matches_plain(form):
    """idx = arange(M) must give exactly the plain GEMM on the same rows, with the
    same kernel form (forms differ in how the K sum is split: two issuers'
    partial sums, one chain per pair)."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.random_problem(21, 300, 400, 264, dtype="bf16", with_c=True, alpha=0.5)
    plain = run(p)
    p.idx = torch.arange(300, dtype=torch.int32)
    gathered = run(p)
    assert torch.equal(plain, gathered)


def test_gather_duplicates_identical_rows():
    p = workloads.random_problem(22, 256, 300, 200, dtype="f16", gather_rows=50)
    p.idx[:] = torch.from_numpy(np.random.default_rng(1).integers(0, 4, 256).astype(np.int32))
    D = run(p).cpu()
    for r in range(4):
        rows = (p.idx == r).nonzero().flatten()
        assert all(torch.equal(D[rows[0]], D[k]) for k in rows)
    ref, absprod, _ = oracle_full(p)
    assert_within(D, ref, absprod, p.out, "duplicates")


def test_gather_bad_index_reports_and_zeroes():
    p = workloads.random_problem(23, 130, 96, 64, dtype="bf16", with_c=True, beta=0.5,
                                 gather_rows=40)
    p.idx[3] = 40
    p.idx[129] = -7
    D = run(p)
    assert device_status() == binding.GEMM_ERR_INDEX
    ref, absprod, bad = oracle_full(p)
    assert bad
    assert_within(D, ref, absprod, p.out, "bad index")
    assert torch.equal(D[3].cpu(), 0.5 * p.C[3])


def test_c_absent_equals_zero_c():
    p = workloads.random_problem(24, 200, 300, 128, dtype="bf16", alpha=1.5)
    D0 = run(p)
    p.C = torch.zeros((200, 300))
    Dz = run(p)
    assert torch.equal(D0, Dz)


def test_beta_zero_does_not_read_c():
    p = workloads.random_problem(25, 130, 70, 64, dtype="bf16", beta=0.0)
    D0 = run(p)
    p.C = torch.full((130, 70), float("nan"))
    assert torch.equal(run(p), D0)


def test_in_place_d_is_c():
    p = workloads.random_problem(26, 260, 300, 136, dtype="f16", values="quarter",
                                 with_c=True, alpha=0.5, beta=2.0)
    ref, _, _ = oracle_full(p)
    C = p.C.to(DEV)
    D = binding.gemm_f16(p.A.to(DEV), p.B.to(DEV), C, C, alpha=0.5, beta=2.0)
    assert D.data_ptr() == C.data_ptr()
    assert_bits(D, ref, OUT_F32, "in place")


def test_k_zero_gives_beta_c():
    C = torch.randn(70, 90)
    A = torch.empty((70, 0), dtype=torch.bfloat16)
    B = torch.empty((90, 0), dtype=torch.bfloat16)
    D = binding.gemm_bf16(A.to(DEV), B.to(DEV), C.to(DEV), alpha=3.0, beta=0.5)
    assert torch.equal(D.cpu(), 0.5 * C)
    D2 = binding.gemm_bf16(A.to(DEV), B.to(DEV))
    assert torch.count_nonzero(D2) == 0


def test_empty_m_n_is_noop():
    A = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((5, 64), dtype=torch.bfloat16, device=DEV)
    assert binding.gemm_bf16(A, B).shape == (0, 5)
    assert binding.gemm_bf16(B, A).shape == (5, 0)


def test_strided_operands():
    """Leading dimensions larger than the logical widths."""
    p = workloads.random_problem(27, 150, 170, 136, dtype="bf16", values="quarter",
                                 with_c=True, alpha=0.5, beta=-1.0)
    ref, _, _ = oracle_full(p)
    Abig = torch.zeros((150, 200), dtype=torch.bfloat16)
    Abig[:, :136] = p.A
    Bbig = torch.zeros((170, 144), dtype=torch.bfloat16)
    Bbig[:, :136] = p.B
    Cbig = torch.zeros((150, 180))
    Cbig[:, :170] = p.C
    Dbig = torch.full((150, 176), 7.0, device=DEV)
    A, B, C = Abig.to(DEV)[:, :136], Bbig.to(DEV)[:, :136], Cbig.to(DEV)[:, :170]
    D = Dbig[:, :170]
    binding.gemm_bf16(A, B, C, D, alpha=0.5, beta=-1.0)
    assert_bits(D, ref, OUT_F32, "strided")
    assert torch.all(Dbig[:, 170:] == 7.0)


def test_wait_timeout_is_reported_and_context_survives():
    """A stage whose expected byte count is never met: the bounded wait runs out,
    the kernel returns GEMM_ERR_TIMEOUT, and the next call works."""
    p = workloads.random_problem(28, 256, 256, 256, dtype="bf16", values="quarter")
    binding.gemm_set_wait_timeout(50_000_000)  # 50 ms
    binding.gemm_debug_inject(1)
    try:
        run(p)
        assert device_status() == binding.GEMM_ERR_TIMEOUT
    finally:
        binding.gemm_debug_inject(0)
        binding.gemm_set_wait_timeout(0)
    ref, _, _ = oracle_full(p)
    assert_bits(run(p), ref, OUT_F32, "after timeout")


def test_host_side_errors_with_device_tensors():
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    D = torch.zeros((64, 64), device=DEV)
    lib = binding.load_library()
    s = binding._stream_ptr(None)
    # misaligned A (offset by one element)
    st = lib.gemm_bf16(64, 64, 64, A.data_ptr() + 2, 64, B.data_ptr(), 64, None, 0,
                       D.data_ptr(), 64, 0, 1.0, 0.0, s)
    assert st == 2
    # D overlapping A
    st = lib.gemm_bf16(32, 32, 64, A.data_ptr(), 64, B.data_ptr(), 64, None, 0,
                       A.data_ptr(), 64, 0, 1.0, 0.0, s)
    assert st == 4


SKINNY_SHAPES = [(1, 3000, 640), (5, 1000, 520), (16, 4096, 1024), (17, 777, 264),
                 (33, 2048, 4096), (64, 5000, 136), (64, 128, 640), (2, 28672, 4096)]


@pytest.mark.parametrize("M,N,K", SKINNY_SHAPES)
@pytest.mark.parametrize("form", [(2, 0), (0, 0)], ids=["skinny", "auto"])
def test_skinny_quarter_bit_exact(M, N, K, form):
    """M <= 64 through the swap-AB stream-K kernel (forced), and through whatever
    the automatic choice gives the shape; exact inputs stay exact through the
    skinny kernel's split partial sums."""
    binding.gemm_debug_force_tile(*form)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = binding.gemm_query_plan(M, N, K, sm_count=sms)
    assert plan.kernel == 2 or form == (0, 0)
    for out, with_c, alpha, beta in [(OUT_F32, True, 0.5, 2.0), (OUT_BF16, False, 1.0, 0.0)]:
        p = workloads.random_problem(M + N + K, M, N, K, dtype="bf16", values="quarter",
                                     with_c=with_c, alpha=alpha, beta=beta, out=out)
        ref, _, _ = oracle_full(p)
        assert_bits(run(p), ref, out, f"kernel {plan.kernel} {M}x{N}x{K} out={out}")


@pytest.mark.parametrize("M,N,K", [(16, 28672, 4096), (40, 3000, 2056), (7, 513, 8192)])
@pytest.mark.parametrize("form", [(2, 0), (0, 0)], ids=["skinny", "auto"])
def test_skinny_normal_within_tolerance(M, N, K, form):
    binding.gemm_debug_force_tile(*form)
    p = workloads.random_problem(M * N + K, M, N, K, dtype="f16", with_c=True, alpha=0.5,
                                 beta=1.0, b_scale=0.02)
    ref, absprod, _ = oracle_full(p)
    assert_within(run(p), ref, absprod, OUT_F32, f"form {form} {M}x{N}x{K}")


def test_skinny_repeated_calls_are_deterministic():
    """The stream-K partial sums are added in a fixed order: identical bits every call."""
    p = workloads.random_problem(31, 16, 8192, 4096, dtype="bf16", with_c=True, alpha=0.5)
    first = run(p)
    for _ in range(3):
        assert torch.equal(run(p), first)


def test_skinny_timeout_is_reported():
    p = workloads.random_problem(32, 16, 2048, 1024, dtype="bf16", values="quarter")
    binding.gemm_debug_force_tile(2, 0)  # (the automatic choice for this shape is the tile kernel)
    binding.gemm_set_wait_timeout(50_000_000)
    binding.gemm_debug_inject(1)
    try:
        run(p)
        assert device_status() == binding.GEMM_ERR_TIMEOUT
    finally:
        binding.gemm_debug_inject(0)
        binding.gemm_set_wait_timeout(0)
    ref, _, _ = oracle_full(p)
    assert_bits(run(p), ref, OUT_F32, "skinny after timeout")


@pytest.mark.parametrize("M", [16, 300])
def test_k_tail_padding_is_not_read(M):
    """K = 20 with a row pitch of 24: the 4 padding columns hold NaN and must not
    reach the result (TMA zero-fills past the tensor's K extent)."""
    K, ld, N = 20, 24, 200
    p = workloads.random_problem(33, M, N, K, dtype="bf16", values="quarter")
    Ap = torch.full((M, ld), float("nan"), dtype=torch.bfloat16)
    Ap[:, :K] = p.A
    Bp = torch.full((N, ld), float("nan"), dtype=torch.bfloat16)
    Bp[:, :K] = p.B
    ref, _, _ = oracle_full(p)
    D = binding.gemm_bf16(Ap.to(DEV)[:, :K], Bp.to(DEV)[:, :K])
    assert_bits(D, ref, OUT_F32, "K tail")
