"""ctypes binding of the C ABI in include/tg_gemm_relu.h.

Argument marshalling only: every step of the computation runs in the library's kernels.
The ``tg_*`` functions keep the C names and signatures (raw pointers as ints, a stream
handle as an int); :func:`gemm_relu` / :func:`gemm_relu_host` are torch/numpy conveniences
over them.  If the shared library has not been built, loading raises — there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))

TG_OK = 0
TG_ERR_INVALID_ARG = 1
TG_ERR_MISALIGNED = 2
TG_ERR_UNSUPPORTED_DEVICE = 3
TG_ERR_CUDA = 4
TG_ERR_TIMEOUT = 5
TG_ERR_NO_WORKSPACE = 6

TG_EPILOGUE_NONE = 0
TG_EPILOGUE_RELU = 1
TG_DEBUG_DROP_FIRST_STAGE = 1


class tg_options(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "block_n", "split_k", "force_repack", "force_workspace", "panel_m", "max_ctas",
        "debug_flags", "timeout_ms", "pair", "tail", "swap_ab", "a_in_place",
        "repack_overlap", "tmem_decode", "dequant_first")]


class tg_epilogue(ctypes.Structure):
    _fields_ = [("activation", ctypes.c_int), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("ldr", ctypes.c_int64)]


TG_ACT_NONE, TG_ACT_RELU, TG_ACT_GELU, TG_ACT_GELU_TANH = 0, 1, 2, 3


class tg_plan(ctypes.Structure):
    _fields_ = [
        ("block_m", ctypes.c_int), ("block_n", ctypes.c_int), ("block_k", ctypes.c_int),
        ("stages", ctypes.c_int), ("split_k", ctypes.c_int),
        ("kblocks", ctypes.c_int64), ("kblocks_per_split", ctypes.c_int64),
        ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64), ("units", ctypes.c_int64),
        ("grid", ctypes.c_int), ("panel_m", ctypes.c_int),
        ("repack_a", ctypes.c_int), ("repack_b", ctypes.c_int),
        ("workspace_epilogue", ctypes.c_int), ("workspace_bytes", ctypes.c_int64),
        ("kernels", ctypes.c_int), ("cta_pair", ctypes.c_int),
        ("tail_tiles", ctypes.c_int64), ("a_row_classes", ctypes.c_int),
        ("repack_overlap", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class TgError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = tg_status_string(status) if _lib is not None else f"status {status}"
        if status == TG_ERR_CUDA and _lib is not None:
            msg += f" (cudaError {tg_last_cuda_error()})"
        super().__init__(f"{where}: {msg}" if where else msg)


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return os.path.join(PKG, "lib", "libtg_gemm_relu.so")


def load_library() -> ctypes.CDLL:
    """Load the compiled library (build it with ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: the CUDA library has not been built "
                               "(run __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(path)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        gemm_args = [vp, vp, vp, i64, i64, i64, i64, i64, i64, ci]
        L.tg_gemm_relu_f16.argtypes = gemm_args + [vp]
        L.tg_gemm_relu_f16_ex.argtypes = gemm_args + [ctypes.POINTER(tg_options), vp]
        L.tg_gemm_relu_f16_host.argtypes = gemm_args + [vp]
        L.tg_gemm_relu_f16_splitk_noalloc.argtypes = gemm_args + [ci, vp]
        L.tg_gemm_f16_epilogue.argtypes = gemm_args[:9] + [ctypes.POINTER(tg_epilogue),
                                                           ctypes.POINTER(tg_options), vp]
        L.tg_gemm_f16_t.argtypes = [ci, ci] + gemm_args[:9] + [ctypes.POINTER(tg_epilogue),
                                                              ctypes.POINTER(tg_options), vp]
        L.tg_relu_backward_f16.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, vp]
        L.tg_gemm_w4a16_f16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, ci,
                                        ctypes.POINTER(tg_epilogue), ctypes.POINTER(tg_options), vp]
        L.tg_gemm_nf4a16_f16.argtypes = L.tg_gemm_w4a16_f16.argtypes
        L.tg_plan_query.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, ci,
                                    ctypes.POINTER(tg_options), ctypes.POINTER(tg_plan)]
        L.tg_device_error_check.argtypes = [ctypes.POINTER(ctypes.c_uint), ci]
        L.tg_status_string.argtypes = [ci]
        L.tg_status_string.restype = ctypes.c_char_p
        L.tg_last_cuda_error.argtypes = [ctypes.POINTER(ci)]
        L.tg_release_workspace.argtypes = []
        L.tg_version.argtypes = []
        for name in ("tg_gemm_relu_f16", "tg_gemm_relu_f16_ex", "tg_gemm_relu_f16_host",
                     "tg_gemm_relu_f16_splitk_noalloc", "tg_gemm_f16_epilogue",
                     "tg_gemm_f16_t", "tg_relu_backward_f16", "tg_gemm_w4a16_f16",
                     "tg_gemm_nf4a16_f16",
                     "tg_plan_query", "tg_device_error_check", "tg_last_cuda_error",
                     "tg_release_workspace", "tg_version"):
            getattr(L, name).restype = ci
        _lib = L
        return L


# ------------------------- C names, same signatures -------------------------

def _opts(options) -> ctypes.POINTER(tg_options) | None:
    if options is None:
        return None
    if isinstance(options, tg_options):
        return ctypes.pointer(options)
    o = tg_options()
    for k, v in dict(options).items():
        if not hasattr(o, k):
            raise KeyError(f"unknown option {k!r}")
        setattr(o, k, int(v))
    return ctypes.pointer(o)


def tg_gemm_relu_f16(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                     ldc: int, epilogue_flag: int, stream: int = 0) -> int:
    return load_library().tg_gemm_relu_f16(A, B, C, M, N, K, lda, ldb, ldc, epilogue_flag,
                                           stream or None)


def tg_gemm_relu_f16_ex(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                        ldc: int, epilogue_flag: int, options=None, stream: int = 0) -> int:
    return load_library().tg_gemm_relu_f16_ex(A, B, C, M, N, K, lda, ldb, ldc, epilogue_flag,
                                              _opts(options), stream or None)


def tg_gemm_f16_epilogue(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                         ldc: int, activation: int = TG_ACT_NONE, bias: int = 0,
                         residual: int = 0, ldr: int = 0, options=None, stream: int = 0) -> int:
    """C = fp16(act(A·B + bias) + residual); bias/residual are device pointers or 0."""
    e = tg_epilogue(activation, bias or None, residual or None, ldr)
    return load_library().tg_gemm_f16_epilogue(A, B, C, M, N, K, lda, ldb, ldc,
                                               ctypes.byref(e), _opts(options), stream or None)


def tg_gemm_f16_t(trans_a: int, trans_b: int, A: int, B: int, C: int, M: int, N: int, K: int,
                  lda: int, ldb: int, ldc: int, activation: int = TG_ACT_NONE, bias: int = 0,
                  residual: int = 0, ldr: int = 0, options=None, stream: int = 0) -> int:
    """C = fp16(act(op(A)·op(B) + bias) + residual), op = transpose when trans_* is 1."""
    e = tg_epilogue(activation, bias or None, residual or None, ldr)
    return load_library().tg_gemm_f16_t(trans_a, trans_b, A, B, C, M, N, K, lda, ldb, ldc,
                                        ctypes.byref(e), _opts(options), stream or None)


def tg_gemm_w4a16_f16(A: int, Wq: int, scales: int, C: int, M: int, N: int, K: int, lda: int,
                      ldq: int, lds: int, ldc: int, group_size: int,
                      activation: int = TG_ACT_NONE, bias: int = 0, residual: int = 0,
                      ldr: int = 0, options=None, stream: int = 0) -> int:
    """C = fp16(epilogue(A · W)) with int4 weights decoded in the kernel (format in the header)."""
    e = tg_epilogue(activation, bias or None, residual or None, ldr)
    return load_library().tg_gemm_w4a16_f16(A, Wq, scales, C, M, N, K, lda, ldq, lds, ldc,
                                            group_size, ctypes.byref(e), _opts(options),
                                            stream or None)


def tg_gemm_nf4a16_f16(A: int, Wq: int, scales: int, C: int, M: int, N: int, K: int, lda: int,
                       ldq: int, lds: int, ldc: int, group_size: int,
                       activation: int = TG_ACT_NONE, bias: int = 0, residual: int = 0,
                       ldr: int = 0, options=None, stream: int = 0) -> int:
    """C = fp16(epilogue(A · W)) with NF4 weights decoded in the kernel (format in the header)."""
    e = tg_epilogue(activation, bias or None, residual or None, ldr)
    return load_library().tg_gemm_nf4a16_f16(A, Wq, scales, C, M, N, K, lda, ldq, lds, ldc,
                                             group_size, ctypes.byref(e), _opts(options),
                                             stream or None)


def tg_relu_backward_f16(dC: int, C: int, dZ: int, M: int, N: int, lddc: int, ldc: int,
                         lddz: int, stream: int = 0) -> int:
    return load_library().tg_relu_backward_f16(dC, C, dZ, M, N, lddc, ldc, lddz, stream or None)


def tg_gemm_relu_f16_host(hA: int, hB: int, hC: int, M: int, N: int, K: int, lda: int,
                          ldb: int, ldc: int, epilogue_flag: int, stream: int = 0) -> int:
    return load_library().tg_gemm_relu_f16_host(hA, hB, hC, M, N, K, lda, ldb, ldc,
                                                epilogue_flag, stream or None)


def tg_gemm_relu_f16_splitk_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, lda: int,
                                    ldb: int, ldc: int, epilogue_flag: int, split_k: int = 0,
                                    stream: int = 0) -> int:
    """Split-K GEMM whose float32 workspace is a fixed array inside the library, for callers
    that must not allocate device memory during the call (limits in the C header)."""
    return load_library().tg_gemm_relu_f16_splitk_noalloc(A, B, C, M, N, K, lda, ldb, ldc,
                                                          epilogue_flag, split_k,
                                                          stream or None)


TG_STATIC_WORKSPACE_BYTES = 64 << 20


def tg_plan_query(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                  num_sms: int, options=None) -> tuple[int, dict]:
    out = tg_plan()
    st = load_library().tg_plan_query(A, B, C, M, N, K, lda, ldb, ldc, num_sms, _opts(options),
                                      ctypes.byref(out))
    return st, out.as_dict()


def tg_device_error_check(clear: bool = True) -> tuple[int, int]:
    w = ctypes.c_uint(0)
    st = load_library().tg_device_error_check(ctypes.byref(w), 1 if clear else 0)
    return st, int(w.value)


def tg_status_string(status: int) -> str:
    return load_library().tg_status_string(status).decode()


def tg_last_cuda_error() -> int:
    v = ctypes.c_int(0)
    load_library().tg_last_cuda_error(ctypes.byref(v))
    return int(v.value)


def tg_release_workspace() -> int:
    return load_library().tg_release_workspace()


def tg_version() -> int:
    return load_library().tg_version()


# ------------------------- torch / numpy conveniences -------------------------

def _check(st: int, where: str):
    if st != TG_OK:
        raise TgError(st, where)


def _row_major_2d(t, name):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit stride along columns)")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def plan(M: int, N: int, K: int, lda=None, ldb=None, ldc=None, num_sms: int = 152,
         options=None, a_ptr: int = 256, b_ptr: int = 256, c_ptr: int = 256) -> dict:
    """The plan the library picks (pure host computation; pointers only matter for alignment)."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    st, p = tg_plan_query(a_ptr, b_ptr, c_ptr, M, N, K, max(lda, 1), max(ldb, 1), max(ldc, 1),
                          num_sms, options)
    _check(st, "tg_plan_query")
    return p


def gemm_relu(A, B, out=None, epilogue: int = TG_EPILOGUE_RELU, stream=None, options=None):
    """C = relu(A @ B) (or A @ B with ``epilogue=TG_EPILOGUE_NONE``) for CUDA fp16 tensors.

    A (M,K) and B (K,N) must be row-major with unit column stride (a leading dimension larger
    than the width is fine); ``out`` may be a row-major (M,N) view.  Runs on ``stream``
    (default: torch's current stream) and returns without synchronising.
    """
    import torch

    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("A and B must be torch.float16")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors (use gemm_relu_host for host arrays)")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif out.shape != (M, N) or out.dtype != torch.float16 or out.device != A.device:
        raise ValueError("out must be an (M, N) float16 tensor on A's device")
    lda = _row_major_2d(A, "A")
    ldb = _row_major_2d(B, "B")
    ldc = _row_major_2d(out, "out")
    s = stream if stream is not None else torch.cuda.current_stream(A.device)
    handle = s.cuda_stream if hasattr(s, "cuda_stream") else int(s)
    with torch.cuda.device(A.device):
        if options is None:
            st = tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                                  max(lda, 1), max(ldb, 1), max(ldc, 1), epilogue, handle)
        else:
            st = tg_gemm_relu_f16_ex(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                                     max(lda, 1), max(ldb, 1), max(ldc, 1), epilogue, options,
                                     handle)
    _check(st, "tg_gemm_relu_f16")
    return out


def gemm_relu_host(A, B, out=None, epilogue: int = TG_EPILOGUE_RELU, stream: int = 0):
    """End-to-end call on host memory (numpy fp16 arrays or CPU torch tensors, ideally
    page-locked): copies in, computes on the current device, copies out, synchronises."""
    import numpy as np

    def as_np(x):
        if hasattr(x, "numpy"):
            return x.numpy()
        return x

    a, b = as_np(A), as_np(B)
    if a.dtype != np.float16 or b.dtype != np.float16:
        raise TypeError("A and B must be float16")
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out_arr = np.empty((M, N), dtype=np.float16)
        ret = out_arr
    else:
        out_arr = as_np(out)
        ret = out
    for x, n in ((a, "A"), (b, "B"), (out_arr, "out")):
        if x.ndim != 2 or (x.shape[1] > 1 and x.strides[1] != 2):
            raise ValueError(f"{n} must be a row-major 2-D array")
    lda = a.strides[0] // 2 if M > 1 else max(K, 1)
    ldb = b.strides[0] // 2 if K > 1 else max(N, 1)
    ldc = out_arr.strides[0] // 2 if M > 1 else max(N, 1)
    st = tg_gemm_relu_f16_host(a.ctypes.data, b.ctypes.data, out_arr.ctypes.data, M, N, K,
                               max(lda, 1), max(ldb, 1), max(ldc, 1), epilogue, stream)
    _check(st, "tg_gemm_relu_f16_host")
    return ret
