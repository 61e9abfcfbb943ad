"""Checks that pin the oracle to facts other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something the pages or the mathematics fix.  They run against the real oracle
in test_oracle_pins.py and against deliberately broken copies of oracle.c in
test_oracle_mutants.py (where at least one pin must fail).
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
from tensor_core_gemm_02_gb300 import workloads


def _f64(t):
    """Library widening of an f16/bf16 tensor to float64 (torch/numpy, not the oracle)."""
    return t.to(torch.float64).numpy()


def pin_decode_f16():
    # every binary16 pattern against numpy's float16 -> float64 widening
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = oracle.decode(bits, "f16")
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_decode_bf16():
    # every bfloat16 pattern against torch's bfloat16 -> float64 widening
    bits = np.arange(65536, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode(bits, "bf16")
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_worked_example_exact():
    """The "mma.sync" page's worked example: exact rational brute force.

    Entries are quarter-integers, products are multiples of 1/16 and 32 of them
    sum exactly, so the result is a multiple of 1/16 with |value| <= 32.
    """
    p = workloads.worked_16x8x32()
    ref, _, bad = oracle.gemm(p.A, p.B)
    assert not bad
    a = p.A.to(torch.float64).numpy()
    b = p.B.to(torch.float64).numpy()
    for i in range(16):
        for j in range(8):
            exact = sum(Fraction(float(a[i, k])) * Fraction(float(b[j, k])) for k in range(32))
            assert Fraction(float(ref[i, j])) == exact, (i, j)
    assert np.all(np.abs(ref) <= 32)
    assert np.all(ref * 16 == np.round(ref * 16))
    # the page checks against a @ b.T in float32 (rtol = atol = 2e-4)
    np.testing.assert_allclose(ref, p.A.float().numpy() @ p.B.float().numpy().T,
                               rtol=2e-4, atol=2e-4)


def pin_matches_numpy_random_shapes():
    """Non-square shapes catch transposed operands and wrong strides."""
    for seed, (M, N, K) in enumerate([(5, 7, 3), (13, 3, 40), (2, 11, 17), (9, 9, 64), (1, 6, 129)]):
        for dtype in ("f16", "bf16"):
            pr = workloads.random_problem(seed, M, N, K, dtype=dtype, with_c=True,
                                          alpha=0.75, beta=-1.5)
            ref, absprod, bad = oracle.gemm(pr.A, pr.B, pr.C, pr.alpha, pr.beta)
            a, b, c = _f64(pr.A), _f64(pr.B), pr.C.numpy().astype(np.float64)
            want = pr.alpha * (a @ b.T) + pr.beta * c
            tol = 1e-12 * (np.abs(a) @ np.abs(b).T + np.abs(c) + 1)
            assert np.all(np.abs(ref - want) <= tol), (M, N, K, dtype)
            np.testing.assert_allclose(absprod, np.abs(a) @ np.abs(b).T, rtol=1e-12, atol=0)


def pin_two_a_plus_one():
    """The "fma" page's example: with small integers the reference is exactly 2*A+1.

    B = identity (N = K), C = ones, alpha = 2, beta = 1  =>  D = 2 X + 1.
    """
    rng = np.random.default_rng(7)
    K = 24
    X = rng.integers(-64, 65, (10, K)).astype(np.float16)
    eye = np.eye(K, dtype=np.float16)
    ones = np.ones((10, K), np.float32)
    ref, _, _ = oracle.gemm(X, eye, ones, alpha=2.0, beta=1.0)
    assert np.array_equal(ref, 2 * X.astype(np.float64) + 1)


def pin_fma_separation():
    """A case whose exact result lies between float32 neighbours of a rounded multiply.

    acc = 1 + 2^-12, alpha = 1 + 2^-12, C = -1, beta = 1:
    alpha * acc + C = 2^-11 + 2^-24 exactly (fused, one rounding); a rounded
    multiply first gives 1 + 2^-11 (tie to even) and then 2^-11.
    """
    K = 8
    a = np.zeros((1, K), np.float16)
    a[0, 0], a[0, 1] = 1.0, 2.0 ** -12
    b = np.zeros((1, K), np.float16)
    b[0, 0], b[0, 1] = 1.0, 1.0
    c = np.full((1, 1), -1.0, np.float32)
    alpha = float(np.float32(1 + 2.0 ** -12))
    ref, _, _ = oracle.gemm(a, b, c, alpha=alpha, beta=1.0)
    fused = 2.0 ** -11 + 2.0 ** -24
    assert ref[0, 0] == fused
    assert np.float32(ref[0, 0]) == np.float32(fused)
    unfused = np.float32(np.float32(alpha) * np.float32(1 + 2.0 ** -12)) - np.float32(1)
    assert unfused == np.float32(2.0 ** -11) != np.float32(fused)


def pin_alpha_beta_c_cases():
    pr = workloads.random_problem(11, 6, 5, 32, dtype="bf16", values="quarter", with_c=True)
    a, b, c = _f64(pr.A), _f64(pr.B), pr.C.numpy().astype(np.float64)
    # alpha = 0 leaves beta * C exactly
    ref, _, _ = oracle.gemm(pr.A, pr.B, pr.C, alpha=0.0, beta=2.0)
    assert np.array_equal(ref, 2.0 * c)
    # C absent equals an explicit zero C
    r0, _, _ = oracle.gemm(pr.A, pr.B, None, alpha=1.0, beta=1.0)
    rz, _, _ = oracle.gemm(pr.A, pr.B, np.zeros((6, 5), np.float32), alpha=1.0, beta=1.0)
    assert np.array_equal(r0, rz)
    assert np.array_equal(r0, a @ b.T)  # exact on quarter-integers
    # beta = 0 means C is not read: NaN in C does not reach the result
    cn = np.full((6, 5), np.nan, np.float32)
    rn, _, _ = oracle.gemm(pr.A, pr.B, cn, alpha=1.0, beta=0.0)
    assert np.array_equal(rn, a @ b.T)
    # alpha = -1, beta = 0.5, all exact
    rs, _, _ = oracle.gemm(pr.A, pr.B, pr.C, alpha=-1.0, beta=0.5)
    assert np.array_equal(rs, -(a @ b.T) + 0.5 * c)


def pin_gather_invariants():
    rng = np.random.default_rng(5)
    pr = workloads.random_problem(12, 9, 7, 20, dtype="bf16", with_c=True)
    table = pr.A  # 9 x 20
    plain, _, _ = oracle.gemm(table, pr.B, pr.C, 1.0, 1.0)
    ar = torch.arange(9, dtype=torch.int32)
    g, _, bad = oracle.gemm(table, pr.B, pr.C, 1.0, 1.0, idx=ar)
    assert not bad and np.array_equal(g, plain)
    perm = rng.permutation(9).astype(np.int32)
    g2, _, _ = oracle.gemm(table, pr.B, None, 1.0, 0.0, idx=torch.from_numpy(perm))
    want, _, _ = oracle.gemm(table[torch.from_numpy(perm).long()].contiguous(), pr.B, None, 1.0, 0.0)
    assert np.array_equal(g2, want)
    dup = torch.tensor([3, 3, 0, 3], dtype=torch.int32)
    g3, _, _ = oracle.gemm(table, pr.B, None, 1.0, 0.0, idx=dup)
    assert np.array_equal(g3[0], g3[1]) and np.array_equal(g3[0], g3[3])
    assert np.array_equal(g3[0], plain[3] - pr.C.numpy()[3].astype(np.float64))
    # an index outside the table makes the row zero and is reported
    badidx = torch.tensor([1, 9, -1, 2], dtype=torch.int32)
    c4 = pr.C[:4].contiguous()
    g4, _, bad4 = oracle.gemm(table, pr.B, c4, 1.0, 0.5, idx=badidx)
    assert bad4
    assert np.array_equal(g4[1], 0.5 * c4.numpy()[1].astype(np.float64))
    assert np.array_equal(g4[2], 0.5 * c4.numpy()[2].astype(np.float64))


def pin_entries_match_rows():
    pr = workloads.random_problem(13, 17, 19, 40, dtype="f16", with_c=True, alpha=0.5,
                                  beta=2.0)
    full, fabs_, _ = oracle.gemm(pr.A, pr.B, pr.C, pr.alpha, pr.beta)
    ii = np.array([0, 16, 5, 7, 16], np.int64)
    jj = np.array([0, 18, 3, 18, 0], np.int64)
    e, eabs, _ = oracle.gemm_entries(pr.A, pr.B, ii, jj, pr.C, pr.alpha, pr.beta)
    assert np.array_equal(e, full[ii, jj]) and np.array_equal(eabs, fabs_[ii, jj])
    part, _, _ = oracle.gemm(pr.A, pr.B, pr.C, pr.alpha, pr.beta, rows=(4, 11))
    assert np.array_equal(part, full[4:11])


def pin_scatter_rows():
    """Row-scattered form: closed forms that tell the A row (source i) from
    the C row (destination idx[i]), brute force on exact inputs, the identity
    index, and the bad-index and placement rules."""
    rng = np.random.default_rng(11)
    M, K, d_rows = 5, 8, 7
    perm = rng.permutation(d_rows)[:M].astype(np.int32)  # distinct, not the identity
    assert not np.array_equal(perm, np.arange(M))
    c = rng.standard_normal((d_rows, K)).astype(np.float32)
    # A = 0: each row sent is beta * C[destination]
    zeros = torch.zeros((M, K), dtype=torch.float16)
    eye = torch.eye(K, dtype=torch.float16)
    r0, _, bad0 = oracle.scatter_rows(zeros, eye, perm, d_rows, c, alpha=3.0, beta=0.5)
    assert not bad0 and np.array_equal(r0, 0.5 * c[perm].astype(np.float64))
    # B = I, no C: each row sent is alpha * A[source]
    a = torch.from_numpy(rng.integers(-4, 5, (M, K)).astype(np.float32) / 4).to(torch.float16)
    r1, _, _ = oracle.scatter_rows(a, eye, perm, d_rows, None, alpha=-2.0)
    assert np.array_equal(r1, -2.0 * _f64(a))
    # exact brute force against numpy on quarter-integer inputs
    b = torch.from_numpy(rng.integers(-4, 5, (6, K)).astype(np.float32) / 4).to(torch.bfloat16)
    ab = a.to(torch.bfloat16)
    cq = (rng.integers(-4, 5, (d_rows, 6)) / 4).astype(np.float32)
    r2, abs2, _ = oracle.scatter_rows(ab, b, perm, d_rows, cq, alpha=0.5, beta=-1.0)
    assert np.array_equal(r2, 0.5 * (_f64(ab) @ _f64(b).T) - cq[perm].astype(np.float64))
    assert np.array_equal(abs2, np.abs(_f64(ab)) @ np.abs(_f64(b)).T)
    # identity index: the scattered rows are the plain GEMM's rows
    ar = np.arange(M, dtype=np.int32)
    r3, _, _ = oracle.scatter_rows(ab, b, ar, M, cq[:M].copy(), alpha=0.5, beta=-1.0)
    plain, _, _ = oracle.gemm(ab, b, torch.from_numpy(cq[:M].copy()), 0.5, -1.0)
    assert np.array_equal(r3, plain)
    # an index outside [0, d_rows) sends nothing and is reported
    badidx = np.array([2, d_rows, -1, 0, 6], np.int32)
    r4, _, bad4 = oracle.scatter_rows(ab, b, badidx, d_rows, cq, alpha=0.5, beta=-1.0)
    assert bad4 and np.isnan(r4[1]).all() and np.isnan(r4[2]).all()
    want4 = 0.5 * (_f64(ab)[[0, 3, 4]] @ _f64(b).T) - cq[[2, 0, 6]].astype(np.float64)
    assert np.array_equal(r4[[0, 3, 4]], want4)
    # placement: rows named once take the row sent, unnamed rows keep D0,
    # repeated rows are reported with their senders
    d0 = rng.standard_normal((d_rows, 6))
    dup = np.array([4, 1, 4, 9, 0], np.int32)
    placed, rep = oracle.scatter_place(d0, r2, dup)
    assert rep == {4: [0, 2]}
    assert np.array_equal(placed[1], r2[1]) and np.array_equal(placed[0], r2[4])
    for untouched in (2, 3, 5, 6):
        assert np.array_equal(placed[untouched], d0[untouched])
    assert np.isnan(placed[4]).all()


# FP4 E2M1 magnitudes as the OCP MX definition tabulates them (codes 0..7).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _unpack_codes(wq):
    """N x K codes from N x K/2 bytes: even k in the low nibble (numpy, not the oracle)."""
    lo, hi = wq & 15, wq >> 4
    return np.stack([lo, hi], axis=-1).reshape(wq.shape[0], -1)


def _dequant_numpy(wq, ws):
    codes = _unpack_codes(wq).astype(np.int64)
    mag = np.array(E2M1_TABLE)[codes & 7]
    sign = np.where(codes & 8, -1.0, 1.0)
    scale = np.repeat(np.ldexp(1.0, ws.astype(np.int64) - 127), 32, axis=0).T  # N x K
    return sign * mag * scale


def pin_fp4_decode():
    got = oracle.decode_e2m1(np.arange(16))
    want = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    assert np.array_equal(got, want) and np.signbit(got[8]) and not np.signbit(got[0])
    s = np.array([0, 1, 100, 126, 127, 128, 200, 254])
    want_s = np.array([float(Fraction(2) ** (int(v) - 127)) for v in s])
    assert np.array_equal(oracle.decode_ue8m0(s), want_s)
    assert np.isnan(oracle.decode_ue8m0([255])[0])


def pin_w4_matches_numpy():
    rng = np.random.default_rng(13)
    M, N, K = 9, 11, 96
    a = torch.from_numpy(rng.integers(-4, 5, (M, K)).astype(np.float32) / 4).to(torch.bfloat16)
    wq = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    ws = rng.integers(118, 137, (K // 32, N)).astype(np.uint8)
    c = (rng.integers(-4, 5, (M, N)) / 4).astype(np.float32)
    ref, absprod = oracle.w4(a, wq, ws, c, alpha=0.5, beta=-2.0)
    w = _dequant_numpy(wq, ws)
    assert np.array_equal(ref, 0.5 * (_f64(a) @ w.T) - 2.0 * c.astype(np.float64))
    assert np.array_equal(absprod, np.abs(_f64(a)) @ np.abs(w).T)


def pin_w4_nibble_order_and_blocks():
    """A = I picks single weights: W[j][k] lands in D[k][j]."""
    K, N = 64, 3
    a = torch.eye(K, dtype=torch.float16)
    wq = np.zeros((N, K // 2), np.uint8)
    wq[0, 0] = 0x72            # k = 0: code 2 (1.0); k = 1: code 7 (6.0)
    wq[1, 16] = 0x0B           # k = 32: code 11 (-1.5)
    wq[2, 31] = 0x50           # k = 63: code 5 (3.0)
    ws = np.full((K // 32, N), 127, np.uint8)
    ws[1, 1] = 130             # block 1 of row 1: x 8
    ws[1, 2] = 126             # block 1 of row 2: x 0.5
    ref, _ = oracle.w4(a, wq, ws)
    want = np.zeros((K, N))
    want[0, 0], want[1, 0], want[32, 1], want[63, 2] = 1.0, 6.0, -12.0, 1.5
    assert np.array_equal(ref, want)


def _fp4_operand(rng, rows, K, codes=(0, 16), scales=(118, 137)):
    """Packed codes (rows x K/2) and scales (K/32 x rows) drawn from the given ranges."""
    lo = rng.integers(*codes, (rows, K // 2))
    hi = rng.integers(*codes, (rows, K // 2))
    q = (lo | (hi << 4)).astype(np.uint8)
    s = rng.integers(*scales, (K // 32, rows)).astype(np.uint8)
    return q, s


def pin_e2m1_matches_numpy():
    """Both operands FP4: against numpy dequantisation of each and a float64 matmul."""
    rng = np.random.default_rng(17)
    M, N, K = 7, 9, 160
    aq, a_s = _fp4_operand(rng, M, K)
    bq, b_s = _fp4_operand(rng, N, K)
    c = (rng.integers(-4, 5, (M, N)) / 4).astype(np.float32)
    ref, absprod = oracle.e2m1(aq, a_s, bq, b_s, c, alpha=0.5, beta=-2.0)
    a = _dequant_numpy(aq, a_s)
    b = _dequant_numpy(bq, b_s)
    assert np.array_equal(ref, 0.5 * (a @ b.T) - 2.0 * c.astype(np.float64))
    assert np.array_equal(absprod, np.abs(a) @ np.abs(b).T)
    # a row range is the same rows of the full result
    part, _ = oracle.e2m1(aq, a_s, bq, b_s, c, alpha=0.5, beta=-2.0, rows=(2, 5))
    assert np.array_equal(part, ref[2:5])
    # beta = 0 leaves C out (even NaN), C absent likewise
    nan_c = np.full((M, N), np.nan, np.float32)
    r0, _ = oracle.e2m1(aq, a_s, bq, b_s, nan_c, alpha=1.0, beta=0.0)
    r1, _ = oracle.e2m1(aq, a_s, bq, b_s)
    assert np.array_equal(r0, a @ b.T) and np.array_equal(r1, a @ b.T)


def pin_e2m1_identity_picks():
    """One operand the identity (code 2 = 1.0, scale 127) picks single elements of
    the other: D = B^T dequantised (A = I) and D = A dequantised (B = I), with
    scales that differ per row and per 32-element block, so a transposed scale,
    a swapped nibble or a scale shared between the operands shows."""
    K = 64
    eye_q = np.zeros((K, K // 2), np.uint8)
    for k in range(K):
        eye_q[k, k // 2] |= 2 << (4 * (k % 2))
    eye_s = np.full((K // 32, K), 127, np.uint8)
    rng = np.random.default_rng(19)
    xq, xs = _fp4_operand(rng, 5, K, scales=(124, 131))
    want = _dequant_numpy(xq, xs)                        # 5 x K
    d_a, _ = oracle.e2m1(eye_q, eye_s, xq, xs)           # A = I: D = X^T
    assert np.array_equal(d_a, want.T)
    d_b, _ = oracle.e2m1(xq, xs, eye_q, eye_s)           # B = I: D = X
    assert np.array_equal(d_b, want)
    # closed-form spot values: row 0 of X, element 1 (high nibble of byte 0)
    # and element 33 (block 1)
    code1 = int(xq[0, 0]) >> 4
    code33 = int(xq[0, 16]) >> 4
    v = lambda c: (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7]
    assert d_b[0, 1] == v(code1) * 2.0 ** (int(xs[0, 0]) - 127)
    assert d_b[0, 33] == v(code33) * 2.0 ** (int(xs[1, 0]) - 127)


ALL_PINS = [pin_decode_f16, pin_decode_bf16, pin_worked_example_exact,
            pin_matches_numpy_random_shapes, pin_two_a_plus_one, pin_fma_separation,
            pin_alpha_beta_c_cases, pin_gather_invariants, pin_entries_match_rows,
            pin_scatter_rows, pin_fp4_decode, pin_w4_matches_numpy,
            pin_w4_nibble_order_and_blocks, pin_e2m1_matches_numpy, pin_e2m1_identity_picks]
