"""Host-side checks that need no GPU: the library loads, exports every symbol the
header declares, rejects bad arguments before touching CUDA, and plans kernels."""
import ctypes
import os
import re

import pytest

from tensor_core_gemm_02_gb300 import binding
from tensor_core_gemm_02_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tcgemm.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gemm_f16", "gemm_bf16", "gemm_gather_rows", "gemm_scatter_rows",
              "gemm_accumulate", "gemm_seeded", "gemm_bf16_e2m1", "gemm_e2m1",
              "gemm_check_device_status",
              "gemm_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    names = ["GEMM_OK", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_ALIGNMENT", "GEMM_ERR_UNSUPPORTED",
             "GEMM_ERR_ALIAS", "GEMM_ERR_CUDA", "GEMM_ERR_TIMEOUT", "GEMM_ERR_INDEX"]
    for code, name in enumerate(names):
        assert binding.gemm_status_string(code) == name
    assert binding.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses: validation runs before any CUDA call.
A0, B0, C0, D0, I0 = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def call_bf16(lib, M=64, N=64, K=64, A=A0, lda=64, B=B0, ldb=64, C=None, ldc=0, D=D0, ldd=64,
              out=0, alpha=1.0, beta=0.0):
    return lib.gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, out, alpha, beta, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), 1), (dict(K=-5), 1), (dict(out=3), 1), (dict(D=None), 1),
    (dict(A=None), 1), (dict(B=None), 1), (dict(lda=32), 1), (dict(ldb=8), 1),
    (dict(ldd=63), 1), (dict(C=C0, ldc=10, beta=1.0), 1),
    (dict(A=A0 + 8), 2), (dict(B=B0 + 2), 2), (dict(lda=68), 2), (dict(ldb=100), 2),
    (dict(D=D0 + 2), 2), (dict(C=C0 + 2, ldc=64, beta=1.0), 2),
    (dict(M=1 << 31), 3), (dict(K=1 << 32), 3),
    (dict(D=A0 + 64), 4), (dict(D=B0), 4), (dict(C=D0 + 16, ldc=64, beta=1.0), 4),
    (dict(C=D0, ldc=64, beta=1.0, out=1), 4), (dict(C=D0, ldc=72, ldd=64, beta=1.0), 4),
])
def test_invalid_arguments_rejected_without_gpu(lib, kw, code):
    assert call_bf16(lib, **kw) == code


def test_valid_shapes_that_need_no_launch(lib):
    assert call_bf16(lib, M=0) == 0
    assert call_bf16(lib, N=0) == 0
    # C given but beta == 0: C is ignored entirely (even if misaligned / aliasing)
    assert call_bf16(lib, M=0, C=D0 + 3, beta=0.0) == 0


def test_gather_argument_checks(lib):
    f = lib.gemm_gather_rows
    ok = dict(M=64, N=64, K=64, bf=1, T=A0, rows=100, lda=64, idx=I0, B=B0, ldb=64, C=None,
              ldc=0, D=D0, ldd=64, out=0, alpha=1.0, beta=0.0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["M"], a["N"], a["K"], a["bf"], a["T"], a["rows"], a["lda"], a["idx"], a["B"],
                 a["ldb"], a["C"], a["ldc"], a["D"], a["ldd"], a["out"], a["alpha"], a["beta"],
                 None)

    assert call(idx=None) == 1
    assert call(rows=0) == 1
    assert call(bf=2) == 1
    assert call(idx=I0 + 2) == 2
    assert call(D=I0) == 4  # D overlaps idx
    assert call(D=A0 + 99 * 128) == 4  # D overlaps the last table row


def test_scatter_argument_checks(lib):
    f = lib.gemm_scatter_rows
    ok = dict(M=64, N=64, K=64, bf=1, A=A0, lda=64, B=B0, ldb=64, idx=I0, d_rows=100, C=None,
              ldc=0, D=D0, ldd=64, out=0, alpha=1.0, beta=0.0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["M"], a["N"], a["K"], a["bf"], a["A"], a["lda"], a["B"], a["ldb"], a["idx"],
                 a["d_rows"], a["C"], a["ldc"], a["D"], a["ldd"], a["out"], a["alpha"],
                 a["beta"], None)

    assert call(idx=None) == 1
    assert call(d_rows=0) == 1
    assert call(d_rows=-3) == 1
    assert call(bf=2) == 1
    assert call(d_rows=1 << 31) == 3
    assert call(idx=I0 + 2) == 2
    assert call(D=I0 - 64 * 4 * 99) == 4  # the last of D's 100 rows overlaps idx
    assert call(D=A0 + 63 * 128) == 4  # D overlaps the last row of A
    # C spans d_rows rows like D: the exact in-place form is allowed, a shifted C is not
    assert call(C=D0 + 64 * 4 * 99, ldc=64, beta=1.0) == 4
    assert call(M=0, idx=None) == 0  # nothing to do


def test_accumulate_argument_checks(lib):
    f = lib.gemm_accumulate

    def call(M=64, N=64, K=64, bf=1, A=A0, lda=64, B=B0, ldb=64, D=D0, ldd=64, alpha=1.0):
        return f(M, N, K, bf, A, lda, B, ldb, D, ldd, alpha, None)

    assert call(D=None) == 1
    assert call(bf=2) == 1
    assert call(ldd=63) == 1
    assert call(D=D0 + 2) == 2
    assert call(D=A0 + 64) == 4
    assert call(D=B0) == 4
    assert call(M=0) == 0
    assert call(K=0) == 0  # adds nothing, launches nothing


def test_seeded_argument_checks(lib):
    f = lib.gemm_seeded

    def call(M=64, N=64, K=64, bf=1, A=A0, lda=64, B=B0, ldb=64, C=C0, ldc=64, D=D0, ldd=64,
             out=0):
        return f(M, N, K, bf, A, lda, B, ldb, C, ldc, D, ldd, out, None)

    assert call(C=None) == 1
    assert call(bf=2) == 1
    assert call(ldc=10) == 1
    assert call(C=C0 + 2) == 2
    assert call(C=D0 + 16) == 4
    assert call(M=0, C=None) == 0
    # M <= 64 takes the tile kernel (the skinny kernel has no seeded form)
    assert binding.gemm_query_plan(16, 28672, 4096, seeded=True, sm_count=148).kernel == 1
    assert binding.gemm_query_plan(16, 8, 32, seeded=True, sm_count=148).kernel == 10


def test_fp4_argument_checks(lib):
    f = lib.gemm_bf16_e2m1
    S0 = 0x60000000

    def call(M=16, N=256, K=128, A=A0, lda=128, Bq=B0, ldq=64, Bs=S0, lds=256, C=None, ldc=0,
             D=D0, ldd=256, out=0):
        return f(M, N, K, A, lda, Bq, ldq, Bs, lds, C, ldc, D, ldd, out, 1.0, 0.0, None)

    assert call(Bs=None) == 1
    assert call(ldq=32) == 1            # < K / 2
    assert call(lds=128) == 1           # < N
    assert call(K=48, lda=64) == 3      # not a multiple of 32
    assert call(ldq=72) == 2            # not a multiple of 16 bytes
    # (an unaligned scale base or pitch is fine: the library copies the scales)
    assert call(D=B0 + 64) == 4         # D overlaps the codes
    assert call(D=S0 + 16) == 4         # D overlaps the scales
    assert call(M=0) == 0
    # M <= 64: the skinny kernel with converter warps; more rows: the bf16 plan
    p = binding.gemm_query_plan(16, 28672, 4096, fp4=True, sm_count=148)
    assert (p.kernel, p.bm) == (2, 16) and p.stages > 0
    assert binding.gemm_query_plan(16, 8, 64, fp4=True, sm_count=148).kernel == 2  # never tiny
    assert binding.gemm_query_plan(4096, 4096, 4096, fp4=True, sm_count=148).kernel == 4
    # 64 < M <= 128: two launches of the 64-row skinny kernel
    p = binding.gemm_query_plan(100, 28672, 4096, fp4=True, sm_count=148)
    assert (p.kernel, p.bm) == (2, 64)
    assert binding.gemm_query_plan(129, 28672, 4096, fp4=True, sm_count=148).kernel != 2


def test_e2m1_argument_checks(lib):
    """Both operands FP4: every rule of gemm_e2m1's contract is checked before any
    CUDA call (fake device addresses)."""
    f = lib.gemm_e2m1
    ok = dict(M=128, N=256, K=256, Aq=A0, ldaq=128, As=I0, ldas=128, Bq=B0, ldbq=128, Bs=C0,
              ldbs=256, C=None, ldc=0, D=D0, ldd=256, out=0, alpha=1.0, beta=0.0, image=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["M"], a["N"], a["K"], a["Aq"], a["ldaq"], a["As"], a["ldas"], a["Bq"],
                 a["ldbq"], a["Bs"], a["ldbs"], a["C"], a["ldc"], a["D"], a["ldd"], a["out"],
                 a["alpha"], a["beta"], a["image"], None)

    assert call(M=0) == 0 and call(N=0) == 0            # nothing to do
    assert call(M=-1) == 1 and call(image=2) == 1 and call(out=5) == 1
    assert call(Aq=None) == 1 and call(As=None) == 1 and call(Bs=None) == 1
    assert call(ldaq=64) == 1 and call(ldbq=100) == 1   # shorter than K / 2 bytes
    assert call(ldas=100) == 1 and call(ldbs=255) == 1  # scale rows shorter than M / N
    assert call(K=48) == 3                              # not whole 32-element blocks
    assert call(image=1, K=160, ldaq=96, ldbq=96) == 3  # the 16U4 image: K % 128
    assert call(Aq=A0 + 8) == 2 and call(ldbq=136) == 2  # 16-byte rules of the packed form
    assert call(image=1, Aq=A0 + 16) == 2               # the 16U4 image: 32-byte origins
    assert call(image=1, ldaq=144) == 2                 # and 32-byte strides
    assert call(D=A0 + 64) == 4 and call(D=I0) == 4 and call(D=C0) == 4  # D over Aq, As, Bs
    assert call(C=D0 + 16, ldc=256, beta=1.0) == 4
    assert call(M=1 << 31) == 3


def test_e2m1_plan(lib):
    """gemm_e2m1: M <= 64 with packed codes on the skinny kernel (15); otherwise single
    CTAs (11 packed codes, 12 the 16U4 image), 256 wide unless 128-wide tiles take
    fewer waves; CTA pairs with 256 x 256 tiles (13 / 14) when forced; forced forms
    apply to gemm_e2m1 alone."""
    p = binding.gemm_query_plan(8192, 8192, 8192, e2m1=0, sm_count=148)
    assert (p.kernel, p.bn, p.bm, p.grid, p.stages) == (11, 256, 128, 148, 3)
    p = binding.gemm_query_plan(8192, 8192, 8192, e2m1=1, sm_count=148)
    assert (p.kernel, p.bm) == (12, 128)
    binding.gemm_debug_force_tile(13, 256)
    try:
        p = binding.gemm_query_plan(8192, 8192, 8192, e2m1=0, sm_count=148)
        assert (p.kernel, p.bn, p.bm, p.grid, p.stages) == (13, 256, 256, 148, 5)
    finally:
        binding.gemm_debug_force_tile(0, 0)
    p = binding.gemm_query_plan(16, 28672, 4096, e2m1=1, sm_count=148)
    assert (p.kernel, p.bn, p.tiles, p.grid) == (12, 256, 112, 112)  # the 16U4 image: tiles
    p = binding.gemm_query_plan(16, 28672, 4096, e2m1=0, sm_count=148)
    assert (p.kernel, p.bm, p.bn, p.tiles, p.grid) == (15, 16, 128, 224, 148)  # packed: skinny
    assert binding.gemm_query_plan(33, 1024, 512, e2m1=0, sm_count=148).kernel == 15
    assert binding.gemm_query_plan(64, 1024, 512, e2m1=0, sm_count=148).kernel == 15
    assert binding.gemm_query_plan(65, 1024, 512, e2m1=0, sm_count=148).kernel == 11
    binding.gemm_debug_force_tile(15, 128)
    try:  # forced, the skinny form still takes at most 64 rows
        assert binding.gemm_query_plan(65, 1024, 512, e2m1=0, sm_count=148).kernel == 11
    finally:
        binding.gemm_debug_force_tile(0, 0)
    assert binding.gemm_query_plan(16, 1024, 0, e2m1=0, sm_count=148).kernel == 11  # K == 0
    p = binding.gemm_query_plan(1024, 1024, 1024, e2m1=0, sm_count=148)
    assert (p.kernel, p.bn, p.tiles) == (11, 128, 64)  # single CTAs, the narrower tile
    binding.gemm_debug_force_tile(11, 256)
    try:  # a forced tile form takes small M too
        assert binding.gemm_query_plan(16, 28672, 4096, e2m1=0, sm_count=148).kernel == 11
    finally:
        binding.gemm_debug_force_tile(0, 0)
    binding.gemm_debug_force_tile(11, 128)
    try:
        assert binding.gemm_query_plan(8192, 8192, 8192, e2m1=0, sm_count=148).bn == 128
        assert binding.gemm_query_plan(8192, 8192, 8192, sm_count=148).kernel == 4  # not bf16's
    finally:
        binding.gemm_debug_force_tile(0, 0)
    binding.gemm_debug_force_tile(14, 256)
    try:
        p = binding.gemm_query_plan(300, 200, 256, e2m1=1, sm_count=148)
        assert (p.kernel, p.bm, p.tiles, p.grid) == (14, 256, 2, 4)
    finally:
        binding.gemm_debug_force_tile(0, 0)
    assert binding.gemm_query_plan(0, 8, 32, e2m1=0, sm_count=148).kernel == 0


def test_plan_matches_the_dispatch_rules(lib):
    p = binding.gemm_query_plan(8192, 8192, 8192, sm_count=148)
    assert (p.kernel, p.bm, p.bn, p.grid) == (4, 256, 512, 148)
    assert p.tiles == 32 * 16
    p = binding.gemm_query_plan(8192, 28672, 4096, has_c=True, sm_count=148)
    assert (p.kernel, p.bm, p.bn) == (3, 256, 256) and p.tiles == 32 * 112
    p = binding.gemm_query_plan(8192, 8192, 0, sm_count=148)  # K == 0: single CTAs
    assert p.kernel == 1
    p = binding.gemm_query_plan(1024, 1024, 1024, sm_count=148)
    assert (p.kernel, p.bn) == (1, 64) and p.tiles == 128 and p.grid == 128
    p = binding.gemm_query_plan(16, 28672, 4096, sm_count=148)
    assert (p.kernel, p.bm, p.bn, p.tiles, p.grid) == (2, 16, 128, 224, 148)
    # stream-K shares of 224 * 64 k-blocks over 148 CTAs: at most 2 per tile
    assert p.splits == 2
    p = binding.gemm_query_plan(16384, 4096, 4096, gather=True, sm_count=148)
    assert (p.kernel, p.bm, p.bn, p.grid) == (9, 256, 512, 144) and p.tiles == 64 * 8
    p = binding.gemm_query_plan(16384, 1024, 4096, gather=True, sm_count=148)
    assert (p.kernel, p.bn) == (7, 512)
    p = binding.gemm_query_plan(16384, 4096, 1024, gather=True, sm_count=148)
    assert (p.kernel, p.bn) == (6, 256)
    p = binding.gemm_query_plan(16384, 1024, 1024, gather=True, sm_count=148)
    assert (p.kernel, p.bn) == (5, 256)
    p = binding.gemm_query_plan(16384, 512, 4096, gather=True, sm_count=148)
    assert p.kernel == 4 and p.bn == 512
    # scattered rows: the same shape takes 256 x 256 pairs (the epilogue must overlap)
    p = binding.gemm_query_plan(16384, 4096, 4096, scatter=True, sm_count=148)
    assert (p.kernel, p.bn) == (3, 256)
    p = binding.gemm_query_plan(16384, 4096, 4096, sm_count=148)
    assert (p.kernel, p.bn) == (4, 512)
    p = binding.gemm_query_plan(16, 28672, 4096, scatter=True, sm_count=148)
    assert p.kernel == 2
    plan = binding.Plan()
    assert lib.gemm_query_plan(64, 64, 64, 8, 0, 148, ctypes.byref(plan)) == 1
    p = binding.gemm_query_plan(100, 8192, 8192, sm_count=148)
    assert (p.kernel, p.bn) == (1, 64)
    # 16 < M <= 64: the tile kernel unless K is long against N
    assert binding.gemm_query_plan(40, 1000, 64, sm_count=148).kernel == 1
    assert binding.gemm_query_plan(64, 28672, 4096, sm_count=148).kernel != 2
    assert binding.gemm_query_plan(32, 4096, 4096, sm_count=148).kernel == 2  # K >= N, N K > 2^21
    assert binding.gemm_query_plan(32, 16384, 2048, sm_count=148).kernel != 2
    assert binding.gemm_query_plan(32, 1024, 1024, sm_count=148).kernel != 2  # N K <= 2^21
    assert binding.gemm_query_plan(33, 4096, 4096, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(64, 8192, 4096, sm_count=148).kernel != 2  # K < N
    p = binding.gemm_query_plan(32, 4096, 8192, sm_count=148)
    assert (p.kernel, p.bm) == (2, 32)
    p = binding.gemm_query_plan(40, 1024, 8192, sm_count=148)
    assert (p.kernel, p.bm) == (2, 64)
    assert binding.gemm_query_plan(64, 4096, 4096, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(64, 4096, 16384, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(48, 2048, 8192, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(64, 4096, 14336, sm_count=148).kernel == 2
    # the rule's edge: K >= 2N for 17..64 rows, or K >= N when N K > 2^21
    assert binding.gemm_query_plan(17, 1024, 2048, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(32, 1024, 2047, sm_count=148).kernel == 1
    assert binding.gemm_query_plan(33, 1024, 2048, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(64, 1024, 2040, sm_count=148).kernel == 1
    # scattered and accumulating calls follow the same rule; gathered rows never
    assert binding.gemm_query_plan(48, 8192, 4096, scatter=True, sm_count=148).kernel != 2
    assert binding.gemm_query_plan(32, 4096, 4096, scatter=True, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(16, 4096, 4096, scatter=True, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(16, 4096, 4096, gather=True, sm_count=148).kernel != 2
    # the allocation-free entry point always plans the skinny kernel (or the tiny one)
    p = binding.gemm_query_plan(40, 1000, 64, noalloc=True, sm_count=148)
    assert (p.kernel, p.bm) == (2, 64)
    assert binding.gemm_query_plan(16, 8, 32, noalloc=True, sm_count=148).kernel == 10
    assert binding.gemm_query_plan(65, 1000, 64, noalloc=True, sm_count=148).kernel == 0
    assert binding.gemm_query_plan(16, 1000, 0, noalloc=True, sm_count=148).kernel == 0
    assert binding.gemm_query_plan(0, 10, 10).kernel == 0
    # at most 2^20 multiply-adds: the warp-level kernel, one 16 x 8 block per warp
    p = binding.gemm_query_plan(16, 8, 32, sm_count=148)
    assert (p.kernel, p.bm, p.bn, p.tiles, p.grid) == (10, 16, 8, 1, 1)
    p = binding.gemm_query_plan(64, 128, 128, sm_count=148)
    assert (p.kernel, p.tiles, p.grid) == (10, 4 * 16, 16)
    assert binding.gemm_query_plan(128, 128, 128, sm_count=148).kernel == 1
    # M <= 16: the skinny kernel once N * K > 2^21
    assert binding.gemm_query_plan(16, 1024, 1024, sm_count=148).kernel == 1
    assert binding.gemm_query_plan(16, 1024, 2049, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(8, 4096, 4096, sm_count=148).kernel == 2
    assert binding.gemm_query_plan(300, 200, 0, sm_count=148).kernel == 10  # K = 0: beta * C
    assert binding.gemm_query_plan(3000, 2000, 0, sm_count=148).kernel == 1


def _skinny_steps(tiles, nkb, G, whole):
    """Each CTA's linear K blocks in the order the skinny kernel runs them.
    With whole tiles (FP4 B), floor(T / G) waves of tiles (one wave fewer
    when fewer than G / 4 tiles are left over) go whole, tile S + g + G j to
    CTA g, after its contiguous share [W g / G, W (g+1) / G) of the first S
    tiles' W = S nkb blocks (tail piece, head piece, whole tiles between);
    without (bf16 B), S = T."""
    S = tiles
    if whole:
        waves = tiles // G
        S = tiles - waves * G
        if S and waves and 4 * S < G:
            S += G
    W = S * nkb
    steps = []
    for g in range(G):
        lo, hi = W * g // G, W * (g + 1) // G
        b1, b2 = -(-lo // nkb) * nkb, hi // nkb * nkb
        if b1 < hi:
            mine = list(range(lo, b1)) + list(range(b2, hi)) + list(range(b1, b2))
        else:
            mine = list(range(lo, hi))
        for j in range((tiles - S) // G):
            t = S + g + G * j
            mine += list(range(t * nkb, (t + 1) * nkb))
        steps.append(mine)
    return S, steps


def test_skinny_split_arithmetic_covers_every_block():
    """Shared shares and whole tiles cover every K block once, and every shared
    tile's parts fit its workspace slots."""
    cases = [(224, 64, 148), (3, 5, 7), (1, 1, 1), (10, 3, 30), (1000, 7, 152), (4, 8, 148),
             (8, 16, 148), (64, 16, 148), (224, 64, 152), (300, 64, 148), (304, 8, 152),
             (150, 64, 148), (190, 16, 152), (224, 16, 152)]
    for (tiles, nkb, G), whole in [(c, w) for c in cases for w in (False, True)]:
        G = min(G, -(-(tiles * nkb) // 8))  # at least 8 K blocks per CTA
        S, steps = _skinny_steps(tiles, nkb, G, whole)
        assert (tiles - S) % G == 0 and 0 <= S <= tiles
        flat = sorted(x for mine in steps for x in mine)
        assert flat == list(range(tiles * nkb))
        # every CTA's work is balanced to within one K block
        assert max(map(len, steps)) - min(map(len, steps)) <= 1
        owner = {x: g for g, mine in enumerate(steps) for x in mine}
        parts = [len({owner[x] for x in range(t * nkb, (t + 1) * nkb)}) for t in range(tiles)]
        assert all(n == 1 for n in parts[S:])  # whole tiles
        most = max(parts[:S], default=1)
        # bf16 B: 64 K elements per block; FP4 B: 256
        p = binding.gemm_query_plan(16, tiles * 128, nkb * (256 if whole else 64), sm_count=G,
                                    fp4=whole)
        if p.kernel == 2:  # (the smallest bf16 case runs on the warp-level kernel)
            assert p.grid == G and p.splits == most
        else:
            assert not whole
