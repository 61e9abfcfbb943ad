"""Seeded synthetic inputs for the GEMM workloads (host side, CPU tensors).

This module holds none of the GEMM arithmetic: it only draws random numbers and
rounds them to the operand dtypes.  Both the CUDA path's tests/bench and the
oracle consume what it returns; neither side generates inputs on its own.

Recipe (numpy ``default_rng(seed)``, draws in the order listed, the dtype cast
after each draw; float32 -> f16 by numpy ``astype`` and float32 -> bf16 by
torch ``.to(torch.bfloat16)``, both round-to-nearest-even):

  worked_16x8x32   seed 0: a = integers(-4, 5, (16, 32)) / 4, b likewise
                   (8, 32), both f16; no C; fp32 out.  This is the input of the
                   "mma.sync" page's worked example ("Example: a 16x8 result
                   with two K16 issues").
  f16_1024         seed 1: A, B (1024, 1024) N(0,1) -> f16; C (1024, 1024)
                   N(0,1) float32; alpha = beta = 1; fp32 out.
  bf16_8192        seed 2: A (8192, 8192) N(0,1), B (8192, 8192) 0.02 * N(0,1),
                   both -> bf16; no C; bf16 out.
  mlp_8192x28672x4096
                   seed 3: A (8192, 4096) N(0,1), B (28672, 4096) 0.02 * N(0,1)
                   -> bf16; C (8192, 28672) N(0,1) float32; alpha = 0.5,
                   beta = 1; fp32 out.
  skinny_16x28672x4096
                   the same draws; A[:16] and C[:16] (numpy fills row-major, so
                   C[:16] is the first 16 rows of the C draw and only those are
                   drawn).
  gather_16384_of_65536
                   seed 4: table (65536, 4096) N(0,1) -> bf16, idx =
                   integers(0, 65536, 16384) int32 (repeats allowed),
                   B (4096, 4096) 0.02 * N(0,1) -> bf16; no C; fp32 out.
  scatter_16384_into_65536
                   seed 5: A (16384, 4096) N(0,1) -> bf16, idx =
                   permutation(65536)[:16384] int32 (distinct destination
                   rows), B (4096, 4096) 0.02 * N(0,1) -> bf16; no C; fp32 out
                   into D (65536, 4096), whose other rows are left as they were.
                   The row-scattered dual of the gathered workload.
  skinny_accumulate_16x28672x4096
                   the skinny draws; D starts as C[:16] and receives
                   D += 0.5 * A @ B.T (the accumulating form, no C operand).
  fp4_skinny_16x28672x4096
                   seed 6: A (16, 4096) N(0,1) -> bf16; FP4 weights as codes
                   integers(0, 256, (28672, 2048)) uint8 (two E2M1 codes per
                   byte) and scales integers(118, 121, (128, 28672)) uint8
                   (2^-9 .. 2^-7: weights of the size of 0.02 * N(0,1));
                   C (16, 28672) N(0,1) float32; alpha = 0.5, beta = 1; fp32 out.
  e2m1_16x28672x4096
                   seed 7: both operands FP4 (e2m1_problem, values="random"):
                   A (16 x 4096) codes integers(0, 16) per nibble and scales
                   integers(125, 130), B (28672 x 4096) codes likewise and
                   scales integers(118, 121); C (16, 28672) N(0,1) float32;
                   alpha = 0.5, beta = 1; fp32 out.
  e2m1_8192        seed 8: both operands FP4 as above, M = N = K = 8192; no C;
                   bf16 out.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2
OUT_TORCH = {OUT_F32: torch.float32, OUT_BF16: torch.bfloat16, OUT_F16: torch.float16}


@dataclass
class Problem:
    """One GEMM problem: D = alpha * A @ B.T + beta * C, or the gathered form,
    or (scatter = True) the scattered form D[idx[i]] = alpha * A[i] @ B.T +
    beta * C[idx[i]] into a D of d_rows rows."""
    name: str
    A: torch.Tensor                 # M x K operand, or the gather table
    B: torch.Tensor                 # N x K
    C: torch.Tensor | None = None   # M x N float32 (scattered: d_rows x N)
    idx: torch.Tensor | None = None  # int32 rows into A (gathered) or into D (scattered)
    alpha: float = 1.0
    beta: float = 1.0
    out: int = OUT_F32
    meta: dict = field(default_factory=dict)
    scatter: bool = False
    d_rows: int = 0
    D0: torch.Tensor | None = None  # scattered / accumulating forms: D before the call
    accumulate: bool = False        # D += alpha * A @ B.T into float32 D = D0
    Bs: torch.Tensor | None = None  # FP4 weights: B holds codes (N x K/2 uint8), Bs the
                                    # UE8M0 scales (K/32 x N uint8)
    As: torch.Tensor | None = None  # both operands FP4: A holds codes (M x K/2 uint8), As the
                                    # scales (K/32 x M uint8)
    image: int = 0                  # (both FP4) 0 packed codes, 1 the 16U4_ALIGN16B image

    @property
    def fp4(self) -> bool:
        """FP4 weights with bf16 activations (gemm_bf16_e2m1)."""
        return self.Bs is not None and self.As is None

    @property
    def e2m1(self) -> bool:
        """Both operands FP4 (gemm_e2m1)."""
        return self.As is not None

    @property
    def M(self) -> int:
        return int(self.idx.shape[0]) if self.idx is not None else int(self.A.shape[0])

    @property
    def N(self) -> int:
        return int(self.B.shape[0])

    @property
    def K(self) -> int:
        return int(self.A.shape[1]) * (2 if self.As is not None else 1)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _f16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x.astype(np.float16)))


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _cast(x: np.ndarray, dtype: str) -> torch.Tensor:
    return _f16(x) if dtype == "f16" else _bf16(x)


def worked_16x8x32() -> Problem:
    rng = np.random.default_rng(0)
    a = rng.integers(-4, 5, (16, 32)) / 4
    b = rng.integers(-4, 5, (8, 32)) / 4
    return Problem("worked_16x8x32", _f16(a), _f16(b), None, alpha=1.0, beta=0.0,
                   out=OUT_F32)


def f16_1024() -> Problem:
    rng = np.random.default_rng(1)
    A = _f16(rng.standard_normal((1024, 1024), dtype=np.float32))
    B = _f16(rng.standard_normal((1024, 1024), dtype=np.float32))
    C = torch.from_numpy(rng.standard_normal((1024, 1024), dtype=np.float32))
    return Problem("f16_1024", A, B, C, alpha=1.0, beta=1.0, out=OUT_F32)


def bf16_8192() -> Problem:
    rng = np.random.default_rng(2)
    A = _bf16(rng.standard_normal((8192, 8192), dtype=np.float32))
    B = _bf16(0.02 * rng.standard_normal((8192, 8192), dtype=np.float32))
    return Problem("bf16_8192", A, B, None, alpha=1.0, beta=0.0, out=OUT_BF16)


def _mlp_draws(c_rows: int):
    rng = np.random.default_rng(3)
    A = _bf16(rng.standard_normal((8192, 4096), dtype=np.float32))
    B = _bf16(0.02 * rng.standard_normal((28672, 4096), dtype=np.float32))
    C = torch.from_numpy(rng.standard_normal((c_rows, 28672), dtype=np.float32))
    return A, B, C


def mlp_8192x28672x4096() -> Problem:
    A, B, C = _mlp_draws(8192)
    return Problem("mlp_8192x28672x4096", A, B, C, alpha=0.5, beta=1.0, out=OUT_F32)


def skinny_16x28672x4096() -> Problem:
    A, B, C = _mlp_draws(16)
    return Problem("skinny_16x28672x4096", A[:16].contiguous(), B, C, alpha=0.5,
                   beta=1.0, out=OUT_F32)


def gather_16384_of_65536() -> Problem:
    rng = np.random.default_rng(4)
    table = _bf16(rng.standard_normal((65536, 4096), dtype=np.float32))
    idx = torch.from_numpy(rng.integers(0, 65536, 16384).astype(np.int32))
    B = _bf16(0.02 * rng.standard_normal((4096, 4096), dtype=np.float32))
    return Problem("gather_16384_of_65536", table, B, None, idx=idx, alpha=1.0,
                   beta=0.0, out=OUT_F32)


def skinny_accumulate_16x28672x4096() -> Problem:
    A, B, C = _mlp_draws(16)
    return Problem("skinny_accumulate_16x28672x4096", A[:16].contiguous(), B, None, alpha=0.5,
                   beta=0.0, out=OUT_F32, D0=C, accumulate=True)


def fp4_skinny_16x28672x4096() -> Problem:
    rng = np.random.default_rng(6)
    A = _bf16(rng.standard_normal((16, 4096), dtype=np.float32))
    Bq = torch.from_numpy(rng.integers(0, 256, (28672, 2048)).astype(np.uint8))
    Bs = torch.from_numpy(rng.integers(118, 121, (128, 28672)).astype(np.uint8))
    C = torch.from_numpy(rng.standard_normal((16, 28672), dtype=np.float32))
    return Problem("fp4_skinny_16x28672x4096", A, Bq, C, alpha=0.5, beta=1.0, out=OUT_F32, Bs=Bs)


def scatter_16384_into_65536() -> Problem:
    rng = np.random.default_rng(5)
    A = _bf16(rng.standard_normal((16384, 4096), dtype=np.float32))
    idx = torch.from_numpy(rng.permutation(65536)[:16384].astype(np.int32))
    B = _bf16(0.02 * rng.standard_normal((4096, 4096), dtype=np.float32))
    return Problem("scatter_16384_into_65536", A, B, None, idx=idx, alpha=1.0, beta=0.0,
                   out=OUT_F32, scatter=True, d_rows=65536)


def fp4_operand(rng, rows: int, K: int, codes=(0, 16), scales=(118, 121)):
    """Packed E2M1 codes (rows x K/2 uint8; two independent draws per byte, the
    low nibble first) and UE8M0 scales (K/32 x rows uint8) from the ranges."""
    lo = rng.integers(*codes, (rows, K // 2))
    hi = rng.integers(*codes, (rows, K // 2))
    q = torch.from_numpy((lo | (hi << 4)).astype(np.uint8))
    s = torch.from_numpy(rng.integers(*scales, (K // 32, rows)).astype(np.uint8))
    return q, s


def e2m1_problem(seed: int, M: int, N: int, K: int, values: str = "random", with_c: bool = False,
                 alpha: float = 1.0, beta: float = 1.0, out: int = OUT_F32,
                 image: int = 0) -> Problem:
    """Both operands FP4, seeded.  values="exact": codes 0..4 with either sign
    (|value| <= 2) and scales 126..128, so every product is a multiple of 2^-4
    below 16 and every partial sum of K <= 2^16 products is exact in float32;
    C quarter-integers.  values="random": every code, A's scales 125..129
    (values of the size of N(0,1)), B's 118..120 (of 0.02 N(0,1)); C N(0,1).
    Draw order: A's codes, A's scales, B's codes, B's scales, C."""
    rng = np.random.default_rng(seed)
    if values == "exact":
        ca, sa, cb, sb = (0, 5), (126, 129), (0, 5), (126, 129)
    else:
        ca, sa, cb, sb = (0, 16), (125, 130), (0, 16), (118, 121)

    def draw(rows, codes, scales):
        if values == "exact":  # a sign bit drawn apart from the magnitude
            mag = rng.integers(*codes, (rows, K))
            sgn = rng.integers(0, 2, (rows, K)) << 3
            c = mag | sgn
            q = torch.from_numpy((c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8))
            s = torch.from_numpy(rng.integers(*scales, (K // 32, rows)).astype(np.uint8))
            return q, s
        return fp4_operand(rng, rows, K, codes, scales)

    Aq, As = draw(M, ca, sa)
    Bq, Bs = draw(N, cb, sb)
    C = None
    if with_c:
        C = (torch.from_numpy((rng.integers(-4, 5, (M, N)) / 4).astype(np.float32)) if values == "exact"
             else torch.from_numpy(rng.standard_normal((M, N), dtype=np.float32)))
    return Problem(f"e2m1_{values}_{M}x{N}x{K}", Aq, Bq, C, alpha=alpha, beta=beta, out=out,
                   Bs=Bs, As=As, image=image)


def e2m1_16x28672x4096() -> Problem:
    """Both operands FP4, the decode shape: 16 activation rows, FP4 weights of
    the MLP shape, C, alpha = 0.5, fp32 out (seed 7)."""
    p = e2m1_problem(7, 16, 28672, 4096, with_c=True, alpha=0.5, beta=1.0)
    p.name = "e2m1_16x28672x4096"
    return p


def e2m1_8192() -> Problem:
    """Both operands FP4, M = N = K = 8192, no C, bf16 out (seed 8)."""
    p = e2m1_problem(8, 8192, 8192, 8192, alpha=1.0, beta=0.0, out=OUT_BF16)
    p.name = "e2m1_8192"
    return p


WORKLOADS = {
    "worked_16x8x32": worked_16x8x32,
    "f16_1024": f16_1024,
    "bf16_8192": bf16_8192,
    "mlp_8192x28672x4096": mlp_8192x28672x4096,
    "skinny_16x28672x4096": skinny_16x28672x4096,
    "gather_16384_of_65536": gather_16384_of_65536,
    "scatter_16384_into_65536": scatter_16384_into_65536,
    "skinny_accumulate_16x28672x4096": skinny_accumulate_16x28672x4096,
    "fp4_skinny_16x28672x4096": fp4_skinny_16x28672x4096,
    "e2m1_16x28672x4096": e2m1_16x28672x4096,
    "e2m1_8192": e2m1_8192,
}


def random_problem(seed: int, M: int, N: int, K: int, dtype: str = "bf16",
                   values: str = "normal", with_c: bool = False, alpha: float = 1.0,
                   beta: float = 1.0, out: int = OUT_F32, gather_rows: int | None = None,
                   b_scale: float = 1.0, scatter_rows: int | None = None,
                   repeats: bool = False) -> Problem:
    """A seeded problem of any size.

    values="quarter": entries are integers in [-4, 4] divided by 4 (the worked
    example's recipe; C likewise), so every partial sum is exact in float32.
    values="normal": N(0,1) entries (B scaled by b_scale, C N(0,1)).
    gather_rows: if set, A is a table of that many rows and M random indices
    (with repeats) are drawn into it.
    scatter_rows: if set, the scattered form into a D of that many rows: after
    the draws above, idx = M distinct rows (permutation(scatter_rows)[:M]; with
    repeats=True, integers(0, scatter_rows, M)), then C (scatter_rows x N, if
    with_c) and D0 (scatter_rows x N, rounded to the output type).
    """
    rng = np.random.default_rng(seed)
    a_rows = gather_rows if gather_rows is not None else M

    def draw(shape, scale=1.0):
        if values == "quarter":
            return (rng.integers(-4, 5, shape) / 4).astype(np.float32)
        return (scale * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)

    A = _cast(draw((a_rows, K)), dtype)
    idx = None
    if gather_rows is not None:
        idx = torch.from_numpy(rng.integers(0, gather_rows, M).astype(np.int32))
    B = _cast(draw((N, K), b_scale), dtype)
    if scatter_rows is not None:
        if repeats:
            ix = rng.integers(0, scatter_rows, M)
        else:
            ix = rng.permutation(scatter_rows)[:M]
        idx = torch.from_numpy(ix.astype(np.int32))
        C = torch.from_numpy(draw((scatter_rows, N))) if with_c else None
        D0 = torch.from_numpy(draw((scatter_rows, N))).to(OUT_TORCH[out])
        return Problem(f"random_scatter_{values}_{M}x{N}x{K}_{dtype}_into_{scatter_rows}", A,
                       B, C, idx=idx, alpha=alpha, beta=beta, out=out, scatter=True,
                       d_rows=scatter_rows, D0=D0)
    C = torch.from_numpy(draw((M, N))) if with_c else None
    return Problem(f"random_{values}_{M}x{N}x{K}_{dtype}", A, B, C, idx=idx,
                   alpha=alpha, beta=beta, out=out)
