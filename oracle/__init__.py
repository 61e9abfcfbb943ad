"""fp64 CPU oracle for D = alpha * A @ B.T + beta * C (plain, gathered and
scattered forms, FP4 block-scaled weights, and both operands FP4 with block
scales).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``tensor_core_gemm_02_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``oracle.c`` (a plain triple loop in double precision;
its header cites the page sections it follows).  This module only builds that
file with gcc, marshals numpy / torch CPU arrays into it, and spreads rows over
host threads (ctypes releases the GIL during the foreign call).

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the pages fix, closed forms, exact brute force and library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

F16, BF16 = 0, 1
_DTYPES = {"f16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into a shared library (gcc, no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_init.restype = None
    lib.oracle_decode.argtypes = [i32, ctypes.c_uint16]
    lib.oracle_decode.restype = dbl
    lib.oracle_gemm_rows.argtypes = [i64, i64, i64, i64, i32, vp, i64, vp, i64,
                                     vp, i64, vp, i64, dbl, dbl, vp, vp, i64]
    lib.oracle_gemm_rows.restype = i32
    lib.oracle_gemm_entries.argtypes = [i64, vp, vp, i64, i32, vp, i64, vp, i64,
                                        vp, i64, vp, i64, dbl, dbl, vp, vp]
    lib.oracle_gemm_entries.restype = i32
    lib.oracle_scatter_rows.argtypes = [i64, i64, i64, i64, i32, vp, i64, vp, i64,
                                        vp, i64, vp, i64, dbl, dbl, vp, vp, i64]
    lib.oracle_scatter_rows.restype = i32
    lib.oracle_decode_e2m1.argtypes = [i32]
    lib.oracle_decode_e2m1.restype = dbl
    lib.oracle_decode_ue8m0.argtypes = [i32]
    lib.oracle_decode_ue8m0.restype = dbl
    lib.oracle_w4_rows.argtypes = [i64, i64, i64, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64,
                                   dbl, dbl, vp, vp, i64]
    lib.oracle_w4_rows.restype = None
    lib.oracle_e2m1_rows.argtypes = [i64, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                     vp, i64, dbl, dbl, vp, vp, i64]
    lib.oracle_e2m1_rows.restype = None
    lib.oracle_init()
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns the ctypes handle."""
    global _lib
    if path is not None:
        # An explicitly named build of oracle.c (used by the mutation tests,
        # which compile deliberately broken copies) replaces the default one.
        _lib = _bind(ctypes.CDLL(path))
        return _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or (
                os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _as_bits(x, dtype: str | None):
    """Return (uint16 ndarray of raw bits, dtype code) for an f16/bf16 array."""
    mod = type(x).__module__
    if mod.startswith("torch"):
        import torch
        if x.dtype == torch.bfloat16:
            return x.contiguous().view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float16:
            return x.contiguous().numpy().view(np.uint16), F16
        raise TypeError(f"oracle operands must be f16/bf16, got {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    if x.dtype == np.uint16:
        if dtype is None:
            raise TypeError("raw uint16 operands need dtype='f16' or 'bf16'")
        return x, _DTYPES[dtype]
    raise TypeError(f"oracle operands must be f16/bf16, got {x.dtype}")


def _f32(x):
    if x is None:
        return None
    if type(x).__module__.startswith("torch"):
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("C must be float32")
    return x


def _i32(x):
    if x is None:
        return None
    if type(x).__module__.startswith("torch"):
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.int32:
        raise TypeError("idx must be int32")
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def gemm(A, B, C=None, alpha=1.0, beta=1.0, idx=None, dtype=None, threads=None,
         rows=None):
    """Full reference result.

    A: M x K (or the gather table), B: N x K, C: M x N float32 or None,
    idx: int32 row indices (gathered form) or None.  ``rows`` = (i0, i1) limits
    the computation to a row range.  Returns (ref, absprod, bad_index) with
    ref/absprod float64 arrays of shape (i1 - i0, N).
    """
    lib = load()
    a, code_a = _as_bits(A, dtype)
    b, code_b = _as_bits(B, dtype)
    if code_a != code_b:
        raise TypeError("A and B must have the same dtype")
    c, ix = _f32(C), _i32(idx)
    K = a.shape[1]
    if b.shape[1] != K:
        raise ValueError("A and B disagree on K")
    M = ix.shape[0] if ix is not None else a.shape[0]
    N = b.shape[0]
    if c is not None and c.shape != (M, N):
        raise ValueError("C must be M x N")
    i0, i1 = rows if rows is not None else (0, M)
    ref = np.empty((i1 - i0, N), np.float64)
    absprod = np.empty((i1 - i0, N), np.float64)
    nthr = threads or default_threads()
    table_rows = a.shape[0]
    bounds = np.linspace(i0, i1, min(nthr, max(1, i1 - i0)) + 1).astype(np.int64)

    def run(lo, hi):
        if hi <= lo:
            return 0
        lo, hi = int(lo), int(hi)
        off = (lo - i0) * N * 8
        return lib.oracle_gemm_rows(lo, hi, N, K, code_a, _ptr(a), a.shape[1],
                                    _ptr(ix), table_rows, _ptr(b), b.shape[1],
                                    _ptr(c), N, float(alpha), float(beta),
                                    ref.ctypes.data + off, absprod.ctypes.data + off, N)

    with ThreadPoolExecutor(max_workers=nthr) as ex:
        bad = list(ex.map(lambda p: run(*p), zip(bounds[:-1], bounds[1:])))
    return ref, absprod, bool(any(bad))


def gemm_entries(A, B, ii, jj, C=None, alpha=1.0, beta=1.0, idx=None, dtype=None,
                 threads=None):
    """Reference values at selected output coordinates (ii[e], jj[e])."""
    lib = load()
    a, code_a = _as_bits(A, dtype)
    b, code_b = _as_bits(B, dtype)
    if code_a != code_b:
        raise TypeError("A and B must have the same dtype")
    c, ix = _f32(C), _i32(idx)
    ii = np.ascontiguousarray(ii, np.int64)
    jj = np.ascontiguousarray(jj, np.int64)
    n = ii.shape[0]
    K = a.shape[1]
    N = b.shape[0]
    ldc = c.shape[1] if c is not None else N
    ref = np.empty(n, np.float64)
    absprod = np.empty(n, np.float64)
    nthr = threads or default_threads()
    bounds = np.linspace(0, n, min(nthr, max(1, n)) + 1).astype(np.int64)

    def run(lo, hi):
        lo, hi = int(lo), int(hi)
        if hi <= lo:
            return 0
        return lib.oracle_gemm_entries(hi - lo, ii.ctypes.data + lo * 8,
                                       jj.ctypes.data + lo * 8, K, code_a, _ptr(a),
                                       a.shape[1], _ptr(ix), a.shape[0], _ptr(b),
                                       b.shape[1], _ptr(c), ldc, float(alpha),
                                       float(beta), ref.ctypes.data + lo * 8,
                                       absprod.ctypes.data + lo * 8)

    with ThreadPoolExecutor(max_workers=nthr) as ex:
        bad = list(ex.map(lambda p: run(*p), zip(bounds[:-1], bounds[1:])))
    return ref, absprod, bool(any(bad))


def scatter_rows(A, B, idx, d_rows, C=None, alpha=1.0, beta=1.0, dtype=None, threads=None):
    """Rows that a row-scattered GEMM sends: row i (M x N result) is
    alpha * A[i] @ B.T + beta * C[idx[i]], bound for row idx[i] of D.

    C (d_rows x N float32) is indexed by destination row, like D.  Returns
    (rows, absprod, bad_index); a row with an index outside [0, d_rows) is NaN
    and sets bad_index.
    """
    lib = load()
    a, code_a = _as_bits(A, dtype)
    b, code_b = _as_bits(B, dtype)
    if code_a != code_b:
        raise TypeError("A and B must have the same dtype")
    c, ix = _f32(C), _i32(idx)
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("A and B disagree on K")
    if ix is None or ix.shape[0] != M:
        raise ValueError("idx must hold one destination row per row of A")
    if c is not None and c.shape != (d_rows, N):
        raise ValueError("C must be d_rows x N")
    rows = np.empty((M, N), np.float64)
    absprod = np.empty((M, N), np.float64)
    nthr = threads or default_threads()
    bounds = np.linspace(0, M, min(nthr, max(1, M)) + 1).astype(np.int64)

    def run(lo, hi):
        lo, hi = int(lo), int(hi)
        if hi <= lo:
            return 0
        off = lo * N * 8
        return lib.oracle_scatter_rows(lo, hi, N, K, code_a, _ptr(a), a.shape[1], _ptr(ix),
                                       int(d_rows), _ptr(b), b.shape[1], _ptr(c), N,
                                       float(alpha), float(beta), rows.ctypes.data + off,
                                       absprod.ctypes.data + off, N)

    with ThreadPoolExecutor(max_workers=nthr) as ex:
        bad = list(ex.map(lambda p: run(*p), zip(bounds[:-1], bounds[1:])))
    return rows, absprod, bool(any(bad))


def scatter_place(D0, rows, idx):
    """Place the rows a scattered GEMM sends into a copy of D0 (float64).

    Rows of D named by no valid index keep D0.  A row named once holds the
    row sent to it.  A row named more than once is left NaN in the result and
    listed in the returned dict {row: [i, ...]}: every element of it must equal
    the same element of one of the rows sent to it (which one is unspecified).
    """
    D = np.array(D0, np.float64, copy=True)
    ix = np.asarray(idx, np.int64)
    valid = (ix >= 0) & (ix < D.shape[0])
    senders: dict[int, list[int]] = {}
    for i in np.nonzero(valid)[0]:
        senders.setdefault(int(ix[i]), []).append(int(i))
    repeated = {}
    for d, who in senders.items():
        if len(who) == 1:
            D[d] = rows[who[0]]
        else:
            D[d] = np.nan
            repeated[d] = who
    return D, repeated


def decode_e2m1(codes) -> np.ndarray:
    """Value of each FP4 E2M1 code (0..15)."""
    lib = load()
    flat = np.asarray(codes, np.int64).ravel()
    return np.array([lib.oracle_decode_e2m1(int(c)) for c in flat]).reshape(np.shape(codes))


def decode_ue8m0(scales) -> np.ndarray:
    """Value 2^(s - 127) of each UE8M0 scale byte (255: NaN)."""
    lib = load()
    flat = np.asarray(scales, np.int64).ravel()
    return np.array([lib.oracle_decode_ue8m0(int(c)) for c in flat]).reshape(np.shape(scales))


def w4(A, Wq, Ws, C=None, alpha=1.0, beta=1.0, dtype=None, threads=None):
    """alpha * A @ W.T + beta * C with FP4 weights W (N x K) given as packed codes
    Wq (N x K/2 uint8, element k in the low nibble of byte k/2 for even k) and
    UE8M0 scales Ws (K/32 x N uint8).  Returns (ref, absprod) as float64 M x N."""
    lib = load()
    a, code_a = _as_bits(A, dtype)
    wq = np.ascontiguousarray(np.asarray(Wq, np.uint8))
    ws = np.ascontiguousarray(np.asarray(Ws, np.uint8))
    c = _f32(C)
    M, K = a.shape
    N = wq.shape[0]
    if K % 32 or wq.shape[1] != K // 2 or ws.shape != (K // 32, N):
        raise ValueError("Wq must be N x K/2 and Ws K/32 x N, K a multiple of 32")
    ref = np.empty((M, N), np.float64)
    absprod = np.empty((M, N), np.float64)
    nthr = threads or default_threads()
    bounds = np.linspace(0, M, min(nthr, max(1, M)) + 1).astype(np.int64)

    def run(lo, hi):
        lo, hi = int(lo), int(hi)
        if hi > lo:
            off = lo * N * 8
            lib.oracle_w4_rows(lo, hi, N, K, code_a, _ptr(a), a.shape[1], _ptr(wq), wq.shape[1],
                               _ptr(ws), N, _ptr(c), N, float(alpha), float(beta),
                               ref.ctypes.data + off, absprod.ctypes.data + off, N)

    with ThreadPoolExecutor(max_workers=nthr) as ex:
        list(ex.map(lambda p: run(*p), zip(bounds[:-1], bounds[1:])))
    return ref, absprod


def e2m1(Aq, As, Bq, Bs, C=None, alpha=1.0, beta=1.0, threads=None, rows=None):
    """alpha * A @ B.T + beta * C with both operands FP4: packed E2M1 codes Aq
    (M x K/2 uint8) and Bq (N x K/2 uint8), even k in the low nibble, and UE8M0
    block scales As (K/32 x M uint8) and Bs (K/32 x N uint8), one per 32
    elements along K.  ``rows`` = (i0, i1) limits the computation to a row
    range.  Returns (ref, absprod) as float64 arrays of shape (i1 - i0, N)."""
    lib = load()
    aq = np.ascontiguousarray(np.asarray(Aq, np.uint8))
    a_s = np.ascontiguousarray(np.asarray(As, np.uint8))
    bq = np.ascontiguousarray(np.asarray(Bq, np.uint8))
    b_s = np.ascontiguousarray(np.asarray(Bs, np.uint8))
    c = _f32(C)
    M, K = aq.shape[0], 2 * aq.shape[1]
    N = bq.shape[0]
    if K % 32 or bq.shape[1] != K // 2 or a_s.shape != (K // 32, M) or b_s.shape != (K // 32, N):
        raise ValueError("Aq must be M x K/2, Bq N x K/2, As K/32 x M, Bs K/32 x N, "
                         "K a multiple of 32")
    if c is not None and c.shape != (M, N):
        raise ValueError("C must be M x N")
    i0, i1 = rows if rows is not None else (0, M)
    ref = np.empty((i1 - i0, N), np.float64)
    absprod = np.empty((i1 - i0, N), np.float64)
    nthr = threads or default_threads()
    bounds = np.linspace(i0, i1, min(nthr, max(1, i1 - i0)) + 1).astype(np.int64)

    def run(lo, hi):
        lo, hi = int(lo), int(hi)
        if hi > lo:
            off = (lo - i0) * N * 8
            lib.oracle_e2m1_rows(lo, hi, N, K, _ptr(aq), aq.shape[1], _ptr(a_s), M, _ptr(bq),
                                 bq.shape[1], _ptr(b_s), N, _ptr(c), N, float(alpha),
                                 float(beta), ref.ctypes.data + off, absprod.ctypes.data + off, N)

    with ThreadPoolExecutor(max_workers=nthr) as ex:
        list(ex.map(lambda p: run(*p), zip(bounds[:-1], bounds[1:])))
    return ref, absprod


def decode(bits, dtype: str) -> np.ndarray:
    """Decoded double value of each 16-bit pattern (uint16 array)."""
    lib = load()
    code = _DTYPES[dtype]
    flat = np.asarray(bits, np.uint16).ravel()
    out = np.array([lib.oracle_decode(code, int(v)) for v in flat], np.float64)
    return out.reshape(np.shape(bits))
