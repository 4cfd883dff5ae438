"""Oracle for C = relu(A·B): a plain, slow, CPU restatement of the definition.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
leg may import this package.  It shares no code with the CUDA path and never imports it.

The arithmetic lives in ``tg_oracle.c`` (see its header for the passages it follows):
C[i,j] = fp16_rne(relu(sum_k A[i,k]*B[k,j])), sum in float32 in increasing k, plus a
float64-accumulated twin that is the near-exact reference for tolerances.
"""

from __future__ import annotations

import ctypes
import os
import time

import numpy as np

from . import build as _build

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        L.tg_oracle_gemm_relu.restype = ctypes.c_int
        L.tg_oracle_gemm_relu.argtypes = [p, p, i64, i64, i64, i64, i64, p, i64, p, i64,
                                          ctypes.c_int, p, p, p, p, ctypes.c_int]
        L.tg_oracle_f64_to_f16.restype = ctypes.c_uint16
        L.tg_oracle_f64_to_f16.argtypes = [ctypes.c_double]
        L.tg_oracle_f32_to_f16.restype = ctypes.c_uint16
        L.tg_oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.tg_oracle_f16_to_f64.restype = ctypes.c_double
        L.tg_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        for name in ("tg_oracle_f32_to_f16_array", "tg_oracle_f64_to_f16_array",
                     "tg_oracle_f16_to_f64_array"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [p, p, i64]
        L.tg_oracle_gemm_epilogue.restype = ctypes.c_int
        L.tg_oracle_gemm_epilogue.argtypes = [p, p, i64, i64, i64, i64, i64, p, i64, p, i64,
                                              ctypes.c_int, p, p, i64, p, p, p, ctypes.c_int]
        L.tg_oracle_dequant_w4.restype = ctypes.c_int
        L.tg_oracle_dequant_w4.argtypes = [p, p, i64, i64, i64, i64, i64, p]
        L.tg_oracle_dequant_nf4.restype = ctypes.c_int
        L.tg_oracle_dequant_nf4.argtypes = [p, p, i64, i64, i64, i64, i64, p]
        L.tg_oracle_nf4_code.restype = ctypes.c_double
        L.tg_oracle_nf4_code.argtypes = [ctypes.c_int]
        L.tg_oracle_max_threads.restype = ctypes.c_int
        L.tg_oracle_max_threads.argtypes = []
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def f64_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().tg_oracle_f64_to_f16_array(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().tg_oracle_f32_to_f16_array(_ptr(x), _ptr(y), x.size)
    return y


def f16_bits_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, dtype=np.float64)
    lib().tg_oracle_f16_to_f64_array(_ptr(h), _ptr(y), h.size)
    return y


def max_threads() -> int:
    return int(lib().tg_oracle_max_threads())


def gemm_relu(A, B, relu: bool = True, rows=None, cols=None, lda=None, ldb=None, M=None,
              N=None, K=None, want=("f32", "f64"), threads: int = 0) -> dict:
    """relu(A·B) on the rows x cols sub-grid (all of C by default).

    A, B: fp16 arrays, either 2-D (M,K)/(K,N) or flat buffers with explicit M, N, K, lda, ldb.
    Returns a dict with any of: ``out16_f32acc`` / ``acc_f32`` (float32-accumulated result
    bits and pre-relu sums) and ``out16_f64acc`` / ``acc_f64`` (float64-accumulated), each of
    shape (len(rows), len(cols)).
    """
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    if A.dtype not in (np.float16, np.uint16) or B.dtype not in (np.float16, np.uint16):
        raise TypeError("A and B must be fp16 (or their uint16 bit patterns)")
    if A.ndim == 2 and M is None:
        M, K = A.shape
        lda = K if lda is None else lda
    if B.ndim == 2 and N is None:
        N = B.shape[1]
        ldb = N if ldb is None else ldb
    if None in (M, N, K, lda, ldb):
        raise ValueError("flat buffers need M, N, K, lda and ldb")
    if K > 0 and (A.size < (M - 1) * lda + K or B.size < (K - 1) * ldb + N):
        raise ValueError("buffer too small for the given shape and leading dimension")
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    nr, nc = rows.size, cols.size
    res = {}
    o16a = a32 = o16b = a64 = None
    if "f32" in want:
        o16a = res.setdefault("out16_f32acc", np.empty((nr, nc), np.uint16))
        a32 = res.setdefault("acc_f32", np.empty((nr, nc), np.float32))
    if "f64" in want:
        o16b = res.setdefault("out16_f64acc", np.empty((nr, nc), np.uint16))
        a64 = res.setdefault("acc_f64", np.empty((nr, nc), np.float64))
    nullp = ctypes.c_void_p(None)
    rc = lib().tg_oracle_gemm_relu(
        _ptr(A.view(np.uint16)), _ptr(B.view(np.uint16)), M, N, K, lda, ldb,
        _ptr(rows) if nr else nullp, nr, _ptr(cols) if nc else nullp, nc, 1 if relu else 0,
        _ptr(o16a) if o16a is not None else nullp, _ptr(a32) if a32 is not None else nullp,
        _ptr(o16b) if o16b is not None else nullp, _ptr(a64) if a64 is not None else nullp,
        int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return res


ACT = {"none": 0, "relu": 1, "gelu": 2, "gelu_tanh": 3}


def gemm_epilogue(A, B, act="none", bias=None, residual=None, rows=None, cols=None,
                  threads: int = 0) -> dict:
    """fp16(act(A·B + bias) + residual) on the rows x cols sub-grid (all of C by default).

    A (M,K), B (K,N) fp16; bias fp16[N] or None; residual fp16 (M, N) or None.  Returns
    ``out16_f32acc`` and ``out16_f64acc`` (fp16 bits) and ``pre_f64`` (float64 sum + bias,
    before the activation)."""
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    M, K = A.shape
    N = B.shape[1]
    a = ACT[act] if isinstance(act, str) else int(act)
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    nr, nc = rows.size, cols.size
    o32 = np.empty((nr, nc), np.uint16)
    o64 = np.empty((nr, nc), np.uint16)
    pre = np.empty((nr, nc), np.float64)
    nullp = ctypes.c_void_p(None)
    bb = None if bias is None else np.ascontiguousarray(bias, dtype=np.float16).view(np.uint16)
    rr = None if residual is None else np.ascontiguousarray(residual, dtype=np.float16).view(np.uint16)
    if bb is not None and bb.size != N:
        raise ValueError("bias must have N elements")
    ldr = 0 if rr is None else rr.shape[1]
    rc = lib().tg_oracle_gemm_epilogue(
        _ptr(A.view(np.uint16)), _ptr(B.view(np.uint16)), M, N, K, max(K, 1), max(N, 1),
        _ptr(rows) if nr else nullp, nr, _ptr(cols) if nc else nullp, nc, a,
        _ptr(bb) if bb is not None else nullp, _ptr(rr) if rr is not None else nullp, ldr,
        _ptr(o32), _ptr(o64), _ptr(pre), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return {"out16_f32acc": o32, "out16_f64acc": o64, "pre_f64": pre}


def dequant_w4(Wq, scales, K: int, N: int, group: int) -> np.ndarray:
    """fp16 K x N weights from packed int4 Wq (K x ceil(N/8) uint32) and fp16 scales
    (ceil(K/group) x N): w = fp16_rne((q - 8) * s).  See tg_oracle.c for the format."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint32)
    sc = np.ascontiguousarray(scales, dtype=np.float16).view(np.uint16)
    out = np.empty((K, N), np.uint16)
    rc = lib().tg_oracle_dequant_w4(_ptr(Wq), _ptr(sc), K, N, Wq.shape[1], sc.shape[1], group,
                                    _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out.view(np.float16)


def dequant_nf4(Wq, scales, K: int, N: int, group: int) -> np.ndarray:
    """fp16 K x N weights from packed NF4 codes Wq (K x ceil(N/8) uint32, same packing as
    dequant_w4) and fp16 scales (ceil(K/group) x N):
    w = fp16_rne(fp16_rne(nf4[q]) * s), nf4 the QLoRA code table.  See tg_oracle.c."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint32)
    sc = np.ascontiguousarray(scales, dtype=np.float16).view(np.uint16)
    out = np.empty((K, N), np.uint16)
    rc = lib().tg_oracle_dequant_nf4(_ptr(Wq), _ptr(sc), K, N, Wq.shape[1], sc.shape[1], group,
                                     _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out.view(np.float16)


def nf4_codes() -> np.ndarray:
    """The 16 NF4 code values the oracle uses (float64, as printed in QLoRA's Appendix E)."""
    return np.array([lib().tg_oracle_nf4_code(q) for q in range(16)], dtype=np.float64)


def relu_backward(dC, C) -> np.ndarray:
    """dZ = C > 0 ? dC : +0 elementwise, on fp16 arrays (returns fp16 bits).  The relu
    derivative is taken on the forward output C (the practitioner page, section 3.3, asks
    for a hand-written backward behind torch.autograd.Function); -0 and NaN in C count as
    not positive."""
    dC = np.ascontiguousarray(dC, dtype=np.float16)
    C = np.ascontiguousarray(C, dtype=np.float16)
    if dC.shape != C.shape:
        raise ValueError("dC and C must have the same shape")
    with np.errstate(invalid="ignore"):
        pos = C > np.float16(0)
    return np.where(pos, dC.view(np.uint16), np.uint16(0)).astype(np.uint16)


def relu_matmul_backward(A, B, C, dC) -> dict:
    """Gradients of C = relu(A·B) for an incoming dC: dZ = relu_backward(dC, C),
    dA = dZ·B^T and dB = A^T·dZ, each GEMM as the forward oracle (float32 / float64 sums,
    one rounding to fp16).  Transposes are data movement only."""
    dZ = relu_backward(dC, C).view(np.float16)
    dA = gemm_relu(dZ, np.ascontiguousarray(np.asarray(B, np.float16).T), relu=False)
    dB = gemm_relu(np.ascontiguousarray(np.asarray(A, np.float16).T), dZ, relu=False)
    return {"dZ": dZ.view(np.uint16), "dA": dA, "dB": dB}


def timed_rows(A, B, nrows: int, relu: bool = True, threads: int = 0):
    """Time the float32-accumulating oracle on the first ``nrows`` rows of C (a bounded
    sample of the whole product).  Returns (seconds, flops, threads_used)."""
    M, K = A.shape
    N = B.shape[1]
    nrows = max(1, min(nrows, M))
    rows = np.arange(nrows, dtype=np.int64)
    t0 = time.perf_counter()
    gemm_relu(A, B, relu=relu, rows=rows, want=("f32",), threads=threads)
    dt = time.perf_counter() - t0
    return dt, 2.0 * nrows * N * K, (threads if threads > 0 else max_threads())


def cores() -> int:
    return os.cpu_count() or 1
