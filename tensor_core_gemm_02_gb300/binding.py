"""ctypes binding of libtcgemm.so (include/tcgemm.h).  Marshalling only.

The raw entry points keep the C names and argument lists (``lib().gemm_bf16``
etc. via :func:`load_library`).  The functions below take torch CUDA tensors,
read their pointers, leading dimensions and the current stream, call the
C function of the same name and raise :class:`GemmError` on a non-OK status.
Every step of the computation runs in the library's CUDA kernels; there is no
fallback.  If the library is missing this module raises instead of computing
anything some other way.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libtcgemm.so")

GEMM_OK = 0
GEMM_ERR_TIMEOUT = 6
GEMM_ERR_INDEX = 7
OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2
_OUT_OF_DTYPE = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16, torch.float16: OUT_F16}
_DTYPE_OF_OUT = {v: k for k, v in _OUT_OF_DTYPE.items()}

_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__(f"{where}: {gemm_status_string(status)} ({status})")


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("bm", ctypes.c_int32), ("bn", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("tiles", ctypes.c_int64),
                ("splits", ctypes.c_int32), ("grid", ctypes.c_int32)]


def load_library(path: str = LIB_PATH):
    """Load libtcgemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -m tensor_core_gemm_02_gb300.build)")
    lib = ctypes.CDLL(path)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    plain = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, f32, f32, vp]
    lib.gemm_f16.argtypes = plain
    lib.gemm_bf16.argtypes = plain
    lib.gemm_gather_rows.argtypes = [i64, i64, i64, i32, vp, i64, i64, vp, vp, i64, vp, i64,
                                     vp, i64, i32, f32, f32, vp]
    lib.gemm_bf16_e2m1.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                   i32, f32, f32, vp]
    lib.gemm_e2m1.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                              i32, f32, f32, i32, vp]
    lib.gemm_seeded.argtypes = [i64, i64, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64, i32, vp]
    lib.gemm_accumulate.argtypes = [i64, i64, i64, i32, vp, i64, vp, i64, vp, i64, f32, vp]
    lib.gemm_scatter_rows.argtypes = [i64, i64, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64,
                                      vp, i64, i32, f32, f32, vp]
    lib.gemm_skinny_noalloc.argtypes = [i64, i64, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64,
                                        i32, f32, f32, vp]
    lib.gemm_check_device_status.argtypes = [vp]
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_query_plan.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(Plan)]
    lib.gemm_set_wait_timeout.argtypes = [ctypes.c_uint64]
    lib.gemm_debug_inject.argtypes = [i32]
    lib.gemm_debug_force_tile.argtypes = [i32, i32]
    for name in ("gemm_f16", "gemm_bf16", "gemm_gather_rows", "gemm_scatter_rows", "gemm_accumulate",
                 "gemm_seeded", "gemm_bf16_e2m1", "gemm_e2m1",
                 "gemm_skinny_noalloc",
                 "gemm_check_device_status",
                 "gemm_query_plan", "gemm_set_wait_timeout", "gemm_debug_inject",
                 "gemm_debug_force_tile"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ld(t: torch.Tensor) -> int:
    rows, cols = (t.shape[0], t.shape[1]) if t.dim() == 2 else (0, 0)
    if t.dim() != 2 or (cols > 1 and t.stride(1) != 1):
        raise ValueError("matrices must be 2-D with unit column stride")
    if cols == 0:
        return 0  # no columns (K == 0): the leading dimension is never used
    return int(t.stride(0)) if rows > 1 else max(int(t.stride(0)), int(cols))


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _check(status: int, where: str):
    if status != GEMM_OK:
        raise GemmError(status, where)


def _out_tensor(D, M, N, out, device):
    if D is None:
        return torch.empty((M, N), dtype=_DTYPE_OF_OUT[out], device=device)
    if _OUT_OF_DTYPE.get(D.dtype) != out:
        raise TypeError("D's dtype does not match `out`")
    return D


def _plain(name, dtype, A, B, C, D, alpha, beta, out, stream):
    if A.dtype != dtype or B.dtype != dtype:
        raise TypeError(f"{name} needs {dtype} A and B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != (M, N)):
        raise ValueError("C must be float32 M x N")
    D = _out_tensor(D, M, N, out, A.device)
    st = getattr(load_library(), name)(
        M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C) if C is not None else 0,
        _ptr(D), _ld(D), out, float(alpha), float(beta), _stream_ptr(stream))
    _check(st, name)
    return D


def gemm_f16(A, B, C=None, D=None, *, alpha=1.0, beta=1.0, out=OUT_F32, stream=None):
    """D = fma.rn(alpha, A @ B.T, beta * C) with f16 A (M x K) and B (N x K)."""
    return _plain("gemm_f16", torch.float16, A, B, C, D, alpha, beta, out, stream)


def gemm_bf16(A, B, C=None, D=None, *, alpha=1.0, beta=1.0, out=OUT_F32, stream=None):
    """D = fma.rn(alpha, A @ B.T, beta * C) with bf16 A (M x K) and B (N x K)."""
    return _plain("gemm_bf16", torch.bfloat16, A, B, C, D, alpha, beta, out, stream)


def gemm_gather_rows(table, idx, B, C=None, D=None, *, alpha=1.0, beta=1.0, out=OUT_F32,
                     stream=None):
    """D[i] = fma.rn(alpha, table[idx[i]] @ B.T, beta * C[i])."""
    if table.dtype not in (torch.float16, torch.bfloat16) or B.dtype != table.dtype:
        raise TypeError("table and B must both be f16 or both bf16")
    if idx.dtype != torch.int32 or idx.dim() != 1:
        raise TypeError("idx must be a 1-D int32 tensor")
    M = int(idx.shape[0])
    rows, K = table.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("table and B disagree on K")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != (M, N)):
        raise ValueError("C must be float32 M x N")
    D = _out_tensor(D, M, N, out, table.device)
    st = load_library().gemm_gather_rows(
        M, N, K, 1 if table.dtype == torch.bfloat16 else 0, _ptr(table), rows, _ld(table),
        _ptr(idx), _ptr(B), _ld(B), _ptr(C), _ld(C) if C is not None else 0, _ptr(D), _ld(D),
        out, float(alpha), float(beta), _stream_ptr(stream))
    _check(st, "gemm_gather_rows")
    return D


def gemm_scatter_rows(A, B, idx, D, C=None, *, alpha=1.0, beta=1.0, stream=None):
    """D[idx[i]] = fma.rn(alpha, A[i] @ B.T, beta * C[idx[i]]) for every row i of A.

    D (d_rows x N; its dtype picks the output type) is updated in place: rows
    that idx does not name keep their contents.  C, if given, is float32 with
    D's shape (C is D: in-place update of the named rows).  Returns D.
    """
    if A.dtype not in (torch.float16, torch.bfloat16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be f16 or both bf16")
    if idx.dtype != torch.int32 or idx.dim() != 1 or idx.shape[0] != A.shape[0]:
        raise TypeError("idx must be a 1-D int32 tensor with one entry per row of A")
    if D is None or D.dim() != 2:
        raise ValueError("D (the matrix the rows are scattered into) is required")
    out = _OUT_OF_DTYPE.get(D.dtype)
    if out is None:
        raise TypeError("D must be float32, bfloat16 or float16")
    M, K = A.shape
    N = B.shape[0]
    d_rows = int(D.shape[0])
    if B.shape[1] != K or D.shape[1] != N:
        raise ValueError("A, B and D disagree on K or N")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != tuple(D.shape)):
        raise ValueError("C must be float32 with D's shape")
    st = load_library().gemm_scatter_rows(
        M, N, K, 1 if A.dtype == torch.bfloat16 else 0, _ptr(A), _ld(A), _ptr(B), _ld(B),
        _ptr(idx), d_rows, _ptr(C), _ld(C) if C is not None else 0, _ptr(D), _ld(D), out,
        float(alpha), float(beta), _stream_ptr(stream))
    _check(st, "gemm_scatter_rows")
    return D


def gemm_bf16_e2m1(A, Bq, Bs, C=None, D=None, *, alpha=1.0, beta=1.0, out=OUT_F32, stream=None):
    """D = fma.rn(alpha, A @ W.T, beta * C) with bf16 A (M x K) and FP4 weights W
    given as packed E2M1 codes Bq (N x K/2 uint8, even k in the low nibble) and
    UE8M0 block scales Bs (K/32 x N uint8)."""
    if A.dtype != torch.bfloat16:
        raise TypeError("A must be bf16")
    if Bq.dtype != torch.uint8 or Bs.dtype != torch.uint8:
        raise TypeError("Bq and Bs must be uint8")
    M, K = A.shape
    N = Bq.shape[0]
    if Bq.shape[1] * 2 != K or tuple(Bs.shape) != (K // 32, N):
        raise ValueError("Bq must be N x K/2 and Bs K/32 x N")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != (M, N)):
        raise ValueError("C must be float32 M x N")
    D = _out_tensor(D, M, N, out, A.device)
    st = load_library().gemm_bf16_e2m1(
        M, N, K, _ptr(A), _ld(A), _ptr(Bq), _ld(Bq), _ptr(Bs), _ld(Bs), _ptr(C),
        _ld(C) if C is not None else 0, _ptr(D), _ld(D), out, float(alpha), float(beta),
        _stream_ptr(stream))
    _check(st, "gemm_bf16_e2m1")
    return D


FP4_PACKED, FP4_ALIGN16B = 0, 1


def gemm_e2m1(Aq, As, Bq, Bs, C=None, D=None, *, alpha=1.0, beta=1.0, out=OUT_F32,
              image=FP4_PACKED, stream=None):
    """D = fma.rn(alpha, A @ B.T, beta * C) with both operands FP4: packed E2M1
    codes Aq (M x K/2 uint8) and Bq (N x K/2 uint8), even k in the low nibble,
    and UE8M0 block scales As (K/32 x M uint8) and Bs (K/32 x N uint8).
    image: FP4_PACKED (codes as stored, MMA kind::mxf4) or FP4_ALIGN16B (the
    16U4_ALIGN16B load image, MMA kind::mxf8f6f4)."""
    for name, t in (("Aq", Aq), ("As", As), ("Bq", Bq), ("Bs", Bs)):
        if t.dtype != torch.uint8 or t.dim() != 2:
            raise TypeError(f"{name} must be a 2-D uint8 tensor")
    M, K = Aq.shape[0], 2 * Aq.shape[1]
    N = Bq.shape[0]
    if Bq.shape[1] * 2 != K or tuple(As.shape) != (K // 32, M) or tuple(Bs.shape) != (K // 32, N):
        raise ValueError("Aq must be M x K/2, Bq N x K/2, As K/32 x M and Bs K/32 x N")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != (M, N)):
        raise ValueError("C must be float32 M x N")
    D = _out_tensor(D, M, N, out, Aq.device)
    st = load_library().gemm_e2m1(
        M, N, K, _ptr(Aq), _ld(Aq), _ptr(As), _ld(As), _ptr(Bq), _ld(Bq), _ptr(Bs), _ld(Bs),
        _ptr(C), _ld(C) if C is not None else 0, _ptr(D), _ld(D), out, float(alpha), float(beta),
        int(image), _stream_ptr(stream))
    _check(st, "gemm_e2m1")
    return D


def gemm_seeded(A, B, C, D=None, *, out=OUT_F32, stream=None):
    """D = C + A @ B.T with C (float32 M x N) as the accumulator's starting value:
    every K step of the tensor-core sum accumulates onto it."""
    if A.dtype not in (torch.float16, torch.bfloat16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be f16 or both bf16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    if C is None or C.dtype != torch.float32 or tuple(C.shape) != (M, N):
        raise ValueError("C must be float32 M x N")
    D = _out_tensor(D, M, N, out, A.device)
    st = load_library().gemm_seeded(
        M, N, K, 1 if A.dtype == torch.bfloat16 else 0, _ptr(A), _ld(A), _ptr(B), _ld(B),
        _ptr(C), _ld(C), _ptr(D), _ld(D), out, _stream_ptr(stream))
    _check(st, "gemm_seeded")
    return D


def gemm_accumulate(A, B, D, *, alpha=1.0, stream=None):
    """D += alpha * A @ B.T, added into float32 D (M x N) in place.  Returns D."""
    if A.dtype not in (torch.float16, torch.bfloat16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be f16 or both bf16")
    if D is None or D.dtype != torch.float32 or D.dim() != 2:
        raise TypeError("D must be a 2-D float32 tensor")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(D.shape) != (M, N):
        raise ValueError("A, B and D disagree on M, N or K")
    st = load_library().gemm_accumulate(
        M, N, K, 1 if A.dtype == torch.bfloat16 else 0, _ptr(A), _ld(A), _ptr(B), _ld(B),
        _ptr(D), _ld(D), float(alpha), _stream_ptr(stream))
    _check(st, "gemm_accumulate")
    return D


def gemm_skinny_noalloc(A, B, C=None, D=None, *, alpha=1.0, beta=1.0, out=OUT_F32,
                        stream=None):
    """The M <= 64 path with the library's fixed scratch array: the call allocates
    no device memory (D must then be given by the caller to avoid allocating here)."""
    if A.dtype not in (torch.float16, torch.bfloat16) or B.dtype != A.dtype:
        raise TypeError("A and B must both be f16 or both bf16")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != (M, N)):
        raise ValueError("C must be float32 M x N")
    D = _out_tensor(D, M, N, out, A.device)
    st = load_library().gemm_skinny_noalloc(
        M, N, K, 1 if A.dtype == torch.bfloat16 else 0, _ptr(A), _ld(A), _ptr(B), _ld(B),
        _ptr(C), _ld(C) if C is not None else 0, _ptr(D), _ld(D), out, float(alpha),
        float(beta), _stream_ptr(stream))
    _check(st, "gemm_skinny_noalloc")
    return D


def gemm(A, B, C=None, *, alpha=1.0, beta=1.0, out_dtype=torch.float32, D=None, stream=None):
    """Dispatch on A's dtype to gemm_f16 / gemm_bf16."""
    out = _OUT_OF_DTYPE[out_dtype]
    fn = gemm_bf16 if A.dtype == torch.bfloat16 else gemm_f16
    return fn(A, B, C, D, alpha=alpha, beta=beta, out=out, stream=stream)


def gemm_check_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device-side status code."""
    return int(load_library().gemm_check_device_status(_stream_ptr(stream)))


def gemm_query_plan(M, N, K, gather=False, has_c=False, sm_count=148, scatter=False,
                    seeded=False, fp4=False, noalloc=False, e2m1=None) -> Plan:
    """e2m1: None, or FP4_PACKED / FP4_ALIGN16B for gemm_e2m1's plan."""
    p = Plan()
    form = 1 if gather else (2 if scatter else (3 if seeded else (4 if fp4 else (5 if noalloc else 0))))
    if e2m1 is not None:
        form = 6 + int(e2m1)
    _check(load_library().gemm_query_plan(M, N, K, form, int(bool(has_c)),
                                          sm_count, ctypes.byref(p)), "gemm_query_plan")
    return p


def gemm_set_wait_timeout(ns: int) -> None:
    _check(load_library().gemm_set_wait_timeout(int(ns)), "gemm_set_wait_timeout")


def gemm_debug_inject(mode: int) -> None:
    _check(load_library().gemm_debug_inject(int(mode)), "gemm_debug_inject")


def gemm_debug_force_tile(kernel: int, bn: int = 0) -> None:
    _check(load_library().gemm_debug_force_tile(int(kernel), int(bn)), "gemm_debug_force_tile")
