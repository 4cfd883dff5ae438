"""Seeded random shapes through the default plans, against the oracle on sampled rows.

Each case draws M, N and K log-uniformly and checks eight rows of C (the first, the last and
six random ones) against the float64-accumulated oracle with the tolerance and zero rule of
tests/parity.py. The draws cover:
  - relu(A·B) with unaligned leading dimensions and 2-byte-aligned base pointers (the copy paths)
    and with aligned ones (single-CTA, CTA-pair, split-K and tail-split plans);
  - the fused bias / activation / residual epilogue with padded ldc;
  - the int4 and NF4 weight GEMMs with groups of 64 to 256 rows;
  - the transposed-operand GEMM with every combination of stored layouts.
C's padding must come back untouched. Every case is its own test id, so a failure names its
shape."""

import math
import random

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs

from tests.parity import compare
from tests.test_gpu_epilogue import ACT, run as run_epilogue
from tests.test_gpu_parity import run_gpu
from tests.test_gpu_w4 import make, run_w4

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from fp16_gemm_relu_gb300 import build

    build.build()
    torch.cuda.set_device(0)
    yield
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK, f"device error word {word:#x}"


def _logu(rng, lo, hi):
    return int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))


def _rows(rng, M):
    return np.array(sorted({0, M - 1, *(rng.randrange(M) for _ in range(6))}), dtype=np.int64)


def _assert_ok(res, relu, where):
    ok = res["out_of_tol"] == 0 and (not relu or (res["zero_rule"] == 0 and
                                                   res.get("negative_sign", 0) == 0))
    assert ok, f"{where}: {res}"


@pytest.mark.parametrize("i", range(60))
def test_relu_gemm_random_strides(i):
    rng = random.Random(9100 + i)
    while True:
        M, N, K = _logu(rng, 1, 8192), _logu(rng, 1, 8192), _logu(rng, 1, 70000)
        if M * K <= 3e7 and K * N <= 3e7 and M * N <= 3e7:
            break
    odd = rng.random() < 0.5
    lda = K + (rng.choice([1, 2, 3, 5, 7]) if odd else rng.choice([0, 0, 8]))
    ldb = N + (rng.choice([1, 3, 5]) if odd else rng.choice([0, 0, 8]))
    ldc = N + rng.choice([0, 0, 1, 8])
    a_off, b_off, c_off = rng.choice([0, 0, 0, 1]), rng.choice([0, 0, 0, 3]), rng.choice([0, 0, 1])
    relu = rng.random() < 0.8
    a = inputs.tensor(M, K, 9100 + i, 0)
    b = inputs.tensor(K, N, 9100 + i, 1)
    c, pad_ok = run_gpu(a, b, relu, None, lda=lda, ldb=ldb, ldc=ldc, a_off=a_off, b_off=b_off,
                        c_off=c_off)
    where = f"{M}x{N}x{K} lda={lda} ldb={ldb} ldc={ldc} offsets={a_off},{b_off},{c_off}"
    assert pad_ok, where
    rows = _rows(rng, M)
    _assert_ok(compare(c[rows], oracle.gemm_relu(a, b, relu=relu, rows=rows), K, relu), relu,
               where)


@pytest.mark.parametrize("i", range(40))
def test_relu_gemm_random_aligned(i):
    rng = random.Random(9200 + i)
    while True:
        M = _logu(rng, 64, 8192)
        N = -(-_logu(rng, 64, 8192) // 8) * 8
        K = -(-_logu(rng, 64, 32768) // 8) * 8
        if M * K <= 6e7 and K * N <= 6e7 and M * N <= 6e7:
            break
    relu = rng.random() < 0.8
    a = inputs.tensor(M, K, 9200 + i, 0)
    b = inputs.tensor(K, N, 9200 + i, 1)
    c, pad_ok = run_gpu(a, b, relu, None)
    assert pad_ok
    rows = _rows(rng, M)
    _assert_ok(compare(c[rows], oracle.gemm_relu(a, b, relu=relu, rows=rows), K, relu), relu,
               f"{M}x{N}x{K}")


@pytest.mark.parametrize("i", range(40))
def test_epilogue_random(i):
    rng = random.Random(9300 + i)
    while True:
        M, N, K = _logu(rng, 1, 4096), _logu(rng, 1, 4096), _logu(rng, 1, 16384)
        if M * K <= 3e7 and K * N <= 3e7:
            break
    act = rng.choice(list(ACT))
    bias = inputs.tensor(1, N, 9300 + i, 2).ravel() if rng.random() < 0.6 else None
    resid = inputs.tensor(M, N, 9300 + i, 3) if rng.random() < 0.4 else None
    ldc = N + rng.choice([0, 0, 1, 8])
    a = inputs.tensor(M, K, 9300 + i, 0)
    b = inputs.tensor(K, N, 9300 + i, 1)
    got, pad = run_epilogue(a, b, act, bias, resid, None, ldc=ldc)
    where = f"{M}x{N}x{K} ldc={ldc} {act} bias={bias is not None} residual={resid is not None}"
    assert pad.size == 0 or np.isnan(pad.view(np.float16)).all(), where
    rows = _rows(rng, M)
    r = oracle.gemm_epilogue(a, b, act, bias=bias, residual=resid, rows=rows)
    zr = act == "relu" and resid is None
    res = compare(got[rows], {"out16_f64acc": r["out16_f64acc"], "acc_f64": r["pre_f64"]}, K,
                  relu=zr)
    _assert_ok(res, zr, where)


@pytest.mark.parametrize("fmt", ["int4", "nf4"])
@pytest.mark.parametrize("i", range(25))
def test_weight_gemm_random(fmt, i):
    rng = random.Random(9400 + i)
    while True:
        M, N, K = _logu(rng, 1, 2048), _logu(rng, 8, 8192), _logu(rng, 64, 8192)
        if M * K <= 2e7 and K * N <= 4e7:
            break
    G = rng.choice([64, 128, 192, 256])
    act = rng.choice(["none", "relu", "gelu_tanh"])
    a, Wq, S = make(M, N, K, G, 9400 + i)
    got = run_w4(a, Wq, S, N, G, act=ACT[act], fmt=fmt)
    rows = _rows(rng, M)
    w = (oracle.dequant_w4 if fmt == "int4" else oracle.dequant_nf4)(Wq, S, K, N, G)
    r = oracle.gemm_epilogue(a, w, act, rows=rows)
    res = compare(got[rows], {"out16_f64acc": r["out16_f64acc"], "acc_f64": r["pre_f64"]}, K,
                  relu=act == "relu")
    _assert_ok(res, act == "relu", f"{fmt} {M}x{N}x{K} G={G} {act}")


@pytest.mark.parametrize("i", range(32))
def test_transposed_random(i):
    # tg_gemm_f16_t with A and/or B stored transposed (the backward GEMMs' layouts), padded or
    # unaligned leading dimensions, no activation
    from tests.test_gpu_backward import gemm_t

    rng = random.Random(9500 + i)
    while True:
        M, N, K = _logu(rng, 1, 4096), _logu(rng, 1, 4096), _logu(rng, 1, 16384)
        if M * K <= 3e7 and K * N <= 3e7 and M * N <= 3e7:
            break
    ta, tb = i & 1, (i >> 1) & 1
    pad = rng.choice([0, 0, 3, 8])
    a = inputs.tensor(M, K, 9500 + i, 0)
    b = inputs.tensor(K, N, 9500 + i, 1)
    a_st = np.ascontiguousarray(a.T) if ta else a
    b_st = np.ascontiguousarray(b.T) if tb else b
    got = gemm_t(a_st, b_st, ta, tb, M, N, K, None, pad=pad)
    rows = _rows(rng, M)
    _assert_ok(compare(got[rows], oracle.gemm_relu(a, b, relu=False, rows=rows), K, False), False,
               f"ta={ta} tb={tb} {M}x{N}x{K} pad={pad}")
