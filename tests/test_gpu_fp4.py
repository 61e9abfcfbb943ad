"""FP4 weights (E2M1 codes, UE8M0 block scales) on the GPU vs the oracle.

Exact cases: quarter-integer A and scales within 2^-2 .. 2^2 make every product a
multiple of 2^-5 no larger than 24, so K = 4096 sums stay exact in float32 and
results compare bit for bit.  Where no tile's K sum is split over CTAs, the
result must also equal, bit for bit, gemm_bf16 on the dequantised weights.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_bits, assert_within, device_status, run, to_f64
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F32

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    binding.gemm_debug_force_tile(0, 0)
    assert device_status() == binding.GEMM_OK
    yield
    assert device_status() == binding.GEMM_OK


def _problem(seed, M, N, K, values="quarter", smin=125, smax=129, with_c=True, out=OUT_F32,
             alpha=0.5, beta=2.0):
    rng = np.random.default_rng(seed)
    if values == "quarter":
        a = rng.integers(-4, 5, (M, K)) / 4
    else:
        a = rng.standard_normal((M, K))
    A = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    Bq = torch.from_numpy(rng.integers(0, 256, (N, K // 2)).astype(np.uint8))
    Bs = torch.from_numpy(rng.integers(smin, smax + 1, (K // 32, N)).astype(np.uint8))
    C = torch.from_numpy((rng.integers(-4, 5, (M, N)) / 4).astype(np.float32)) if with_c else None
    return workloads.Problem(f"fp4_{M}x{N}x{K}", A, Bq, C, alpha=alpha, beta=beta, out=out, Bs=Bs)


def _ref(p):
    return oracle.w4(p.A, p.B.numpy(), p.Bs.numpy(), p.C, p.alpha, p.beta)


def _dequant_bf16(p):
    """W as bf16 through the oracle's decoders (exact for these scales)."""
    codes = np.stack([p.B.numpy() & 15, p.B.numpy() >> 4], axis=-1).reshape(p.N, -1)
    w = oracle.decode_e2m1(np.arange(16))[codes] * np.repeat(
        oracle.decode_ue8m0(np.arange(256))[p.Bs.numpy()], 32, axis=0).T
    wb = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(wb.double().numpy(), w)
    return wb


@pytest.mark.parametrize("M,N,K", [(1, 300, 64), (16, 1000, 96), (17, 777, 4096),
                                   (33, 2048, 1024), (64, 520, 2048), (16, 28672, 512),
                                   (100, 300, 256), (300, 1000, 1024),
                                   (20, 20000, 1024), (16, 39000, 1024)])
def test_fp4_quarter_bit_exact(M, N, K):
    """Fused skinny path (M <= 64, split K included) and dequantise-then-tile (M > 64).
    On 152 SMs, 20 x 20000 x 1024 shares 78 tiles and gives 79 whole ones to 79
    CTAs (ragged last tile among them); 16 x 39000 x 1024 leaves one tile over two
    whole waves, so one wave more is shared (153 shared, 152 whole)."""
    for out, with_c in [(OUT_F32, True), (OUT_BF16, False)]:
        p = _problem(M * 7 + N + K, M, N, K, with_c=with_c, out=out)
        ref, _ = _ref(p)
        assert_bits(run(p), ref, out, f"fp4 {M}x{N}x{K} out={out}")


@pytest.mark.parametrize("M,N,K", [(16, 4096, 256), (64, 1000, 256), (200, 512, 512)])
def test_fp4_equals_bf16_on_dequantised_weights(M, N, K):
    """M > 64 runs the bf16 kernel itself on the dequantised weights: equal bit
    for bit.  M <= 64 multiplies the same bf16 values, but its MMA issuers each
    sum their own K blocks before the partial sums are added, so the two may
    differ only by float32 reassociation: at most 2 K 2^-24 sum|a||w| (before
    the alpha/beta epilogue, which both apply alike)."""
    p = _problem(M + N, M, N, K, values="normal", smin=112, smax=135)
    got = run(p)
    w = _dequant_bf16(p)
    want = binding.gemm_bf16(p.A.to(DEV), w.to(DEV), p.C.to(DEV), alpha=p.alpha, beta=p.beta)
    if M > 64:
        assert torch.equal(got, want)
        return
    absprod = p.A.double().abs() @ w.double().abs().T
    bound = abs(p.alpha) * 2 * K * 2.0**-24 * absprod + 1e-30
    diff = (got.double().cpu() - want.double().cpu()).abs()
    assert bool((diff <= bound * 1.01 + 2.0**-24 * want.double().cpu().abs()).all())


@pytest.mark.parametrize("smin,smax", [(0, 8), (100, 140), (200, 220)])
def test_fp4_scale_ranges_within_tolerance(smin, smax):
    """Scales from the subnormal 2^-127 up to 2^93; results within the bound."""
    p = _problem(91 + smin, 16, 640, 512, values="normal", smin=smin, smax=smax, beta=1.0)
    ref, absprod = _ref(p)
    assert_within(run(p), ref, absprod, OUT_F32, f"scales {smin}..{smax}")


def test_fp4_nan_scale_gives_nan_columns():
    """Scale 255 is NaN (OCP MX): the columns of W it covers turn the outputs NaN."""
    p = _problem(92, 16, 256, 128, with_c=False)
    p.Bs[1, 7] = 255
    D = run(p).cpu()
    assert torch.isnan(D[:, 7]).all()
    assert not torch.isnan(D[:, 6]).any() and not torch.isnan(D[:, 8]).any()


def test_fp4_strided_operands():
    """Codes and scales with row pitches larger than their rows."""
    p = _problem(93, 24, 300, 256)
    ref, _ = _ref(p)
    Bq_wide = torch.zeros((p.N, 160), dtype=torch.uint8)
    Bq_wide[:, :128] = p.B
    Bs_wide = torch.zeros((p.K // 32, 320), dtype=torch.uint8)
    Bs_wide[:, :300] = p.Bs
    D = binding.gemm_bf16_e2m1(p.A.to(DEV), Bq_wide.to(DEV)[:, :128], Bs_wide.to(DEV)[:, :300],
                               p.C.to(DEV), alpha=p.alpha, beta=p.beta)
    assert_bits(D, ref, OUT_F32, "strided")


def test_fp4_decode_workload_full():
    """16 x 28672 x 4096: the decode step the bench times, every output checked."""
    p = workloads.fp4_skinny_16x28672x4096()
    D = run(p)
    ref, absprod = _ref(p)
    assert_within(D, ref, absprod, OUT_F32, p.name)


def test_fp4_repeated_calls_are_deterministic():
    p = workloads.fp4_skinny_16x28672x4096()
    assert torch.equal(run(p), run(p))
