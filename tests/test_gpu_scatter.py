"""Row-scattered GEMM on the GPU vs the oracle (needs a GB300).

D[idx[i]] = fma.rn(alpha, A[i] @ B.T, beta * C[idx[i]]): rows named once must
match the oracle (bit for bit on quarter-integer inputs), rows named by no
index must keep their contents, and in rows named more than once every element
must be one of the values sent there.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_scatter, device_status, run, to_f64
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


CASES = [("bf16", OUT_F32, True, 0.5, 2.0), ("f16", OUT_BF16, False, 1.0, 0.0),
         ("bf16", OUT_F16, True, -1.0, 1.0), ("f16", OUT_F32, False, 2.0, 0.0)]


@pytest.mark.parametrize("M,N,K,d_rows", [(16, 300, 136, 40), (48, 520, 200, 100),
                                          (129, 257, 72, 500), (300, 520, 264, 700),
                                          (513, 700, 1000, 2000), (256, 96, 64, 256)])
def test_scatter_quarter_bit_exact(M, N, K, d_rows):
    """The automatic choice (warp-level, tile and skinny kernels), ragged
    shapes, every output type."""
    for dtype, out, with_c, alpha, beta in CASES:
        p = workloads.random_problem(M + 7 * N + K, M, N, K, dtype=dtype, values="quarter",
                                     with_c=with_c, alpha=alpha, beta=beta, out=out,
                                     scatter_rows=d_rows)
        assert_scatter(run(p), p, True, f"{M}x{N}x{K} into {d_rows} {dtype} out={out}")


@pytest.mark.parametrize("M,N,K,d_rows", [(16, 300, 136, 40), (48, 520, 200, 100),
                                          (64, 1000, 520, 3000)])
def test_scatter_skinny_forced_bit_exact(M, N, K, d_rows):
    """The skinny kernel's scattered epilogue (forced) on ragged M <= 64 shapes."""
    binding.gemm_debug_force_tile(2, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert binding.gemm_query_plan(M, N, K, scatter=True, sm_count=sms).kernel == 2
    for dtype, out, with_c, alpha, beta in CASES:
        p = workloads.random_problem(M + 9 * N + K, M, N, K, dtype=dtype, values="quarter",
                                     with_c=with_c, alpha=alpha, beta=beta, out=out,
                                     scatter_rows=d_rows)
        assert_scatter(run(p), p, True, f"skinny {M}x{N}x{K} into {d_rows} {dtype} out={out}")


@pytest.mark.parametrize("form", TILE_FORMS, ids=FORM_IDS)
def test_every_tile_form_scatter(form):
    binding.gemm_debug_force_tile(*form)
    for out in (OUT_F32, OUT_BF16):
        p = workloads.random_problem(44, 600, 400, 264, dtype="bf16", values="quarter",
                                     with_c=True, alpha=0.5, out=out, scatter_rows=1500)
        assert_scatter(run(p), p, True, f"scatter form {form} out={out}")


@pytest.mark.parametrize("out", [OUT_F32, OUT_BF16])
def test_scatter_normal_within_tolerance(out):
    p = workloads.random_problem(45, 1000, 520, 320, dtype="bf16", with_c=True, alpha=0.5,
                                 out=out, scatter_rows=3000)
    assert_scatter(run(p), p, False, f"normal out={out}")


def test_scatter_skinny_split_k_exact():
    """M = 16 with enough K blocks that tiles are split over CTAs and reduced."""
    p = workloads.random_problem(46, 16, 4096, 4096, dtype="bf16", values="quarter",
                                 with_c=True, alpha=0.5, scatter_rows=64)
    plan = binding.gemm_query_plan(16, 4096, 4096, has_c=True,
                                   sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan.kernel == 2 and plan.splits > 1
    assert_scatter(run(p), p, True, "skinny split-K")


@pytest.mark.parametrize("form", [(1, 128), (3, 256)], ids=["two_issuers", "pair256"])
def test_scatter_identity_matches_plain(form):
    """idx = arange(M) into a D of M rows gives exactly the plain GEMM (same
    kernel form for both: forms differ in how the K sum is split)."""
    binding.gemm_debug_force_tile(*form)
    p = workloads.random_problem(47, 300, 400, 264, dtype="bf16", with_c=True, alpha=0.5)
    plain = run(p)
    q = workloads.Problem("identity", p.A, p.B, p.C, idx=torch.arange(300, dtype=torch.int32),
                          alpha=p.alpha, beta=p.beta, out=p.out, scatter=True, d_rows=300)
    scattered = run(q)
    assert torch.equal(plain, scattered)


def test_scatter_permutation_matches_plain_rows():
    """A permutation only moves rows: D[perm[i]] equals row i of the plain GEMM
    (tile kernel: the same form for both calls)."""
    binding.gemm_debug_force_tile(1, 128)
    for M in (40, 700):
        p = workloads.random_problem(48 + M, M, 330, 200, dtype="f16", alpha=1.5)
        plain = run(p)
        perm = torch.from_numpy(np.random.default_rng(M).permutation(M).astype(np.int32))
        q = workloads.Problem("perm", p.A, p.B, None, idx=perm, alpha=p.alpha, beta=0.0,
                              out=p.out, scatter=True, d_rows=M)
        scattered = run(q)
        assert torch.equal(scattered[perm.long().to(DEV)], plain)


@pytest.mark.parametrize("M,d_rows", [(256, 40), (20, 8)])
def test_scatter_repeated_targets(M, d_rows):
    p = workloads.random_problem(49, M, 300, 128, dtype="bf16", values="quarter",
                                 with_c=True, beta=0.5, scatter_rows=d_rows, repeats=True)
    assert_scatter(run(p), p, True, "repeated targets")


@pytest.mark.parametrize("M", [130, 33])
def test_scatter_bad_index_reports_and_skips(M):
    """Indices outside D write nothing and set GEMM_ERR_INDEX; other rows are
    exact, rows no valid index names keep their contents."""
    p = workloads.random_problem(50, M, 96, 64, dtype="bf16", values="quarter", with_c=True,
                                 beta=0.5, scatter_rows=400)
    p.idx[3] = 400
    p.idx[M - 1] = -7
    D = run(p)
    assert device_status() == binding.GEMM_ERR_INDEX
    assert_scatter(D, p, True, "bad index")


def test_scatter_in_place_c_is_d():
    """C == D: the named rows are updated in place, D[r] = alpha*acc + beta*D[r]."""
    p = workloads.random_problem(51, 300, 264, 128, dtype="bf16", values="quarter",
                                 alpha=0.5, beta=2.0, scatter_rows=900)
    p.C = p.D0.clone()  # float32, the same values D starts with
    D = p.D0.to(DEV)
    out = binding.gemm_scatter_rows(p.A.to(DEV), p.B.to(DEV), p.idx.to(DEV), D, D,
                                    alpha=p.alpha, beta=p.beta)
    assert out is D
    assert_scatter(D, p, True, "in place")


def test_scatter_unaligned_d_uses_plain_stores():
    """Row pitch of D not a multiple of 16 bytes: the plain-store path."""
    p = workloads.random_problem(52, 200, 130, 96, dtype="f16", values="quarter",
                                 with_c=True, beta=-1.0, scatter_rows=333)
    wide = torch.zeros((333, 131), dtype=torch.float32, device=DEV)
    D = wide[:, :130]
    D.copy_(p.D0.to(DEV))
    run(p, D=D)
    assert_scatter(D, p, True, "ldd = 131")
    assert torch.equal(wide[:, 130].cpu(), torch.zeros(333))


def test_scatter_k_zero_gives_beta_c():
    p = workloads.random_problem(53, 90, 64, 0, dtype="bf16", values="quarter",
                                 with_c=True, beta=0.5, scatter_rows=200)
    assert_scatter(run(p), p, True, "K = 0")


def test_scatter_workload_sampled():
    """16384 rows of N = K = 4096 into a D of 65536 rows, in the launch
    configuration the bench times; sampled rows against the oracle, and the rows
    no index names still zero."""
    p = workloads.scatter_16384_into_65536()
    D = run(p)
    assert device_status() == binding.GEMM_OK
    rng = np.random.default_rng(0)
    pick = np.concatenate([rng.choice(p.M, 48, replace=False), [0, 127, 128, p.M - 1]])
    sub = workloads.Problem("sample", p.A[pick].contiguous(), p.B, None,
                            idx=p.idx[pick].contiguous(), alpha=p.alpha, beta=p.beta,
                            out=p.out, scatter=True, d_rows=p.d_rows)
    rows, absprod, bad = oracle.scatter_rows(sub.A, sub.B, sub.idx, sub.d_rows, None,
                                             sub.alpha, sub.beta)
    assert not bad
    got = to_f64(D[sub.idx.long().to(DEV)])
    err = np.abs(got - rows)
    assert (err <= 2e-3 * absprod + 1e-5).all(), f"max err {err.max()}"
    named = torch.zeros(p.d_rows, dtype=torch.bool)
    named[p.idx.long()] = True
    untouched = torch.nonzero(~named).flatten()[:: 997].to(DEV)
    assert torch.count_nonzero(D[untouched]) == 0
