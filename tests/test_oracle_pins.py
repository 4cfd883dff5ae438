"""Pins for the oracle: each check ties it to something other than itself.

- fp16 rounding against the host compiler's conversion (every 13th binary32 pattern here; all
  2^32 with ``-m slow``) and against numpy's float64 -> float16 conversion;
- hand-derived closed forms (tests/golden/closed_forms.txt);
- exact results: permutation matrices, integer inputs (exact int64 products), rank-one;
- sign invariants (all-negative products), exact rational sums on tiny shapes with the
  float32 recursive-summation error bound, and structural invariants (sub-grid selection,
  leading dimensions, transposition, power-of-two scaling).
A mistake such as a dropped term, a transposed operand, a wrong sign or a wrong summation
order fails at least one of them.
"""

import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def _rne_pin_binary(tmp_path_factory):
    lib = oracle.build.build()
    exe = str(tmp_path_factory.mktemp("pin") / "rne_exhaustive")
    subprocess.run(["gcc", "-O2", "-fopenmp", os.path.join(HERE, "pins", "rne_exhaustive.c"),
                    lib, f"-Wl,-rpath,{os.path.dirname(lib)}", "-lm", "-o", exe], check=True)
    return exe


@pytest.fixture(scope="module")
def rne_exe(tmp_path_factory):
    return _rne_pin_binary(tmp_path_factory)


def test_rne_against_compiler_strided(rne_exe):
    r = subprocess.run([rne_exe, "13"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches f32=0 f64=0" in r.stdout


@pytest.mark.slow
def test_rne_against_compiler_exhaustive(rne_exe):
    r = subprocess.run([rne_exe, "1"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_rne_f64_against_numpy():
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, 200000),
        rng.uniform(-70000, 70000, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, np.inf, -np.inf]),
    ])
    got = oracle.f64_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_decode_all_fp16():
    h = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_bits_to_f64(h)
    want = h.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    # round trip of every non-NaN pattern
    np.testing.assert_array_equal(oracle.f64_to_f16_bits(got[~nan]), h[~nan])


def _golden_cases():
    path = os.path.join(HERE, "golden", "closed_forms.txt")
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if line.startswith("#"):
            continue
        if not line:
            if cur:
                cases.append(cur)
            cur = None
            continue
        key, _, rest = line.partition(" ")
        cur = cur or {}
        cur[key] = rest
    if cur:
        cases.append(cur)
    return cases


def _parse_vals(s):
    out = []
    for t in s.split():
        try:
            out.append(float(t))
        except ValueError:
            out.append(float.fromhex(t))
    return np.array(out, dtype=np.float64)


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["case"])
def test_golden_closed_forms(case):
    M, N, K, relu = (int(v) for v in case["shape"].split())
    A = _parse_vals(case.get("A", "")).astype(np.float16).reshape(M, K)
    B = _parse_vals(case.get("B", "")).astype(np.float16).reshape(K, N)
    # the fixtures only use values that are exact in fp16
    assert np.array_equal(A.astype(np.float64).ravel(), _parse_vals(case.get("A", "")), equal_nan=True)
    res = oracle.gemm_relu(A, B, relu=bool(relu))
    want = np.array([int(t, 16) for t in case["C"].split()], dtype=np.uint16).reshape(M, N)
    np.testing.assert_array_equal(res["out16_f32acc"], want)
    if "acc32" in case:
        acc = _parse_vals(case["acc32"]).astype(np.float32).reshape(M, N)
        np.testing.assert_array_equal(res["acc_f32"], acc)


def test_permutation_is_exact():
    rng = np.random.default_rng(5)
    n, N = 37, 29
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float16)
    P[np.arange(n), perm] = 1.0
    B = inputs.tensor(n, N, 7, 1)
    res = oracle.gemm_relu(P, B)
    want = np.maximum(B[perm].astype(np.float32), 0).astype(np.float16).view(np.uint16)
    want = np.where(want == 0x8000, 0, want)
    for key in ("out16_f32acc", "out16_f64acc"):
        np.testing.assert_array_equal(res[key], want)
    # identity epilogue returns B[perm] bit for bit
    res0 = oracle.gemm_relu(P, B, relu=False)
    np.testing.assert_array_equal(res0["out16_f32acc"], B[perm].view(np.uint16))


@pytest.mark.parametrize("shape", [(33, 47, 129), (64, 64, 1024), (5, 300, 3000)])
def test_integer_inputs_exact(shape):
    M, N, K = shape
    A = inputs.tensor(M, K, 11, 0, "int")
    B = inputs.tensor(K, N, 11, 1, "int")
    exact = A.astype(np.int64) @ B.astype(np.int64)
    assert np.abs(exact).max() < 2 ** 24
    res = oracle.gemm_relu(A, B)
    np.testing.assert_array_equal(res["acc_f32"].astype(np.int64), exact)
    np.testing.assert_array_equal(res["acc_f64"].astype(np.int64), exact)
    want = np.maximum(exact, 0).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(res["out16_f32acc"], want)
    np.testing.assert_array_equal(res["out16_f64acc"], want)
    res0 = oracle.gemm_relu(A, B, relu=False)
    np.testing.assert_array_equal(res0["out16_f32acc"], exact.astype(np.float16).view(np.uint16))


def test_rank_one_closed_form():
    M, N, K = 9, 11, 300
    a = np.arange(-4, 5, dtype=np.float64)                  # M values
    b = np.array([1, -1, 2, -3, 0.5, 0.25, -0.125, 7, -7, 3, -2], dtype=np.float64)
    A = np.repeat(a[:, None], K, axis=1).astype(np.float16)
    B = np.repeat(b[None, :], K, axis=0).astype(np.float16)
    exact = K * np.outer(a, b)                              # exact in float64 and float32
    res = oracle.gemm_relu(A, B)
    np.testing.assert_array_equal(res["acc_f32"], exact.astype(np.float32))
    np.testing.assert_array_equal(res["out16_f32acc"],
                                  np.maximum(exact, 0).astype(np.float16).view(np.uint16))


def test_all_negative_products_give_exact_zero():
    M, N, K = 40, 50, 333
    A = np.abs(inputs.tensor(M, K, 21, 0)) + np.float16(0.01)
    B = -(np.abs(inputs.tensor(K, N, 21, 1)) + np.float16(0.01))
    res = oracle.gemm_relu(A, B)
    assert (res["out16_f32acc"] == 0).all() and (res["out16_f64acc"] == 0).all()
    res0 = oracle.gemm_relu(A, B, relu=False)
    assert (res0["acc_f32"] < 0).all()
    assert (res0["out16_f32acc"] & 0x8000).all()


def _exact_sum(arow, bcol):
    return sum((Fraction(float(x)) * Fraction(float(y)) for x, y in zip(arow, bcol)), Fraction(0))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (7, 5, 17), (3, 17, 64), (4, 4, 129)])
def test_brute_force_exact_rational(M, N, K):
    A = inputs.tensor(M, K, 100 + K, 0)
    B = inputs.tensor(K, N, 100 + K, 1)
    res = oracle.gemm_relu(A, B, relu=False)
    u32 = 2.0 ** -24
    for i in range(M):
        for j in range(N):
            ex = _exact_sum(A[i], B[:, j])
            mag = sum(abs(float(x) * float(y)) for x, y in zip(A[i], B[:, j]))
            # recursive summation in float32: |s - exact| <= (K-1) u sum|a_k b_k| (Higham 2002, 4.2)
            assert abs(Fraction(float(res["acc_f32"][i, j])) - ex) <= Fraction(max(K - 1, 0) * u32 * mag) + Fraction(0)
            assert abs(float(res["acc_f64"][i, j]) - float(ex)) <= max(K - 1, 0) * 2.0 ** -53 * mag
            # the fp64 twin rounds (near-)exactly: fp16 of the exact rational
            want = np.float64(float(ex)).astype(np.float16).view(np.uint16)
            assert res["out16_f64acc"][i, j] == want


def test_subgrid_matches_full_and_leading_dims():
    M, N, K = 45, 70, 91
    A = inputs.tensor(M, K, 31, 0)
    B = inputs.tensor(K, N, 31, 1)
    full = oracle.gemm_relu(A, B)
    rows = np.array([44, 0, 17, 17, 3])
    cols = np.array([5, 69, 0, 33])
    sub = oracle.gemm_relu(A, B, rows=rows, cols=cols)
    for k in ("out16_f32acc", "acc_f32", "out16_f64acc", "acc_f64"):
        np.testing.assert_array_equal(sub[k], full[k][np.ix_(rows, cols)])
    # padded leading dimensions filled with NaN must not leak into the result
    Ap = inputs.embed(A, K + 9, fill=np.nan)
    Bp = inputs.embed(B, N + 3, fill=np.nan)
    pad = oracle.gemm_relu(Ap.ravel(), Bp.ravel(), M=M, N=N, K=K, lda=K + 9, ldb=N + 3)
    for k in ("out16_f32acc", "acc_f32"):
        np.testing.assert_array_equal(pad[k], full[k])


def test_transpose_identity_on_integers():
    M, N, K = 23, 31, 200
    A = inputs.tensor(M, K, 41, 0, "int")
    B = inputs.tensor(K, N, 41, 1, "int")
    c = oracle.gemm_relu(A, B)["out16_f32acc"]
    ct = oracle.gemm_relu(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))["out16_f32acc"]
    np.testing.assert_array_equal(c.T, ct)


def test_power_of_two_scaling():
    M, N, K = 20, 24, 150
    A = inputs.tensor(M, K, 51, 0)
    B = inputs.tensor(K, N, 51, 1)
    r1 = oracle.gemm_relu(A, B, relu=False)
    r2 = oracle.gemm_relu((A.astype(np.float32) * 2).astype(np.float16), B, relu=False)
    np.testing.assert_array_equal(r2["acc_f32"], 2 * r1["acc_f32"])


def test_relu_of_identity_equals_relu_epilogue():
    M, N, K = 30, 40, 77
    A = inputs.tensor(M, K, 61, 0)
    B = inputs.tensor(K, N, 61, 1)
    r0 = oracle.gemm_relu(A, B, relu=False)["out16_f32acc"]
    r1 = oracle.gemm_relu(A, B, relu=True)["out16_f32acc"]
    neg = (r0 & 0x8000) != 0
    np.testing.assert_array_equal(r1, np.where(neg, 0, r0))


def test_rejects_bad_arguments():
    A = np.zeros((2, 3), np.float16)
    B = np.zeros((3, 4), np.float16)
    with pytest.raises(ValueError):
        oracle.gemm_relu(A, B, rows=[2])
    with pytest.raises(ValueError):
        oracle.gemm_relu(A, B, cols=[-1])
