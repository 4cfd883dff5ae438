"""Pins for the oracle's fused epilogue, fp16(act(A·B + bias) + residual).

- With A = 0 the sum is exactly +0, so every output reduces to act(bias[j]) + residual[i, j]:
  checked against Python's own libm (math.erf / math.tanh) and numpy's fp16 rounding.
- GELU at points where the standard normal CDF is tabulated (Phi(1), Phi(2)).
- Integer-valued inputs, bias and residual with relu: exact, so bitwise against int64 numpy.
- The epilogue without bias/residual equals the plain relu / identity oracle bit for bit.
- Both GELUs: act(x) - act(-x) = x (their non-linear part is odd), the tanh form within its
  known 4.7e-4 error of x * Phi(x) computed with erf, and the limits act(0) = 0,
  act(large x) = x, act(very negative x) = 0.  Planted in the oracle on the CPU, a wrong cubic
  coefficient, sqrt(pi/2) for sqrt(2/pi), erf(x/2) for erf(x/sqrt 2) and a dropped tanh term
  each fail at least one of these pins.
"""

import math

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import inputs


def _gelu(x):
    return 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))


def _gelu_tanh(x):
    return 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


ACTS = {"none": lambda x: x, "relu": lambda x: x if x > 0 else 0.0, "gelu": _gelu,
        "gelu_tanh": _gelu_tanh}


@pytest.mark.parametrize("act", list(ACTS))
def test_zero_product_reduces_to_bias_and_residual(act):
    M, N, K = 5, 40, 7
    A = np.zeros((M, K), np.float16)
    B = inputs.tensor(K, N, 3, 1)
    bias = (inputs.tensor(1, N, 4, 0).astype(np.float64) * 6.0).astype(np.float16).ravel()
    res = inputs.tensor(M, N, 5, 1)
    r = oracle.gemm_epilogue(A, B, act, bias=bias, residual=res)
    want = np.array([[ACTS[act](float(bias[j])) + float(res[i, j]) for j in range(N)]
                     for i in range(M)])
    np.testing.assert_array_equal(r["out16_f64acc"], want.astype(np.float16).view(np.uint16))
    np.testing.assert_array_equal(r["pre_f64"], np.broadcast_to(bias.astype(np.float64), (M, N)))


def test_gelu_at_tabulated_normal_cdf():
    # gelu(x) = x * Phi(x); Phi(1) = 0.8413447460685429, Phi(2) = 0.9772498680518208
    A = np.zeros((1, 1), np.float16)
    B = np.zeros((1, 4), np.float16)
    bias = np.array([1.0, -1.0, 2.0, -2.0], np.float16)
    r = oracle.gemm_epilogue(A, B, "gelu", bias=bias)
    want = np.array([0.8413447460685429, -(1 - 0.8413447460685429), 2 * 0.9772498680518208,
                     -2 * (1 - 0.9772498680518208)])
    np.testing.assert_array_equal(r["out16_f64acc"].ravel(), want.astype(np.float16).view(np.uint16))


def test_integer_inputs_with_bias_and_residual_exact():
    M, N, K = 37, 45, 300
    A = inputs.tensor(M, K, 8, 0, "int")
    B = inputs.tensor(K, N, 8, 1, "int")
    bias = inputs.tensor(1, N, 9, 0, "int").ravel() * np.float16(8)
    res = inputs.tensor(M, N, 9, 1, "int")
    exact = A.astype(np.int64) @ B.astype(np.int64) + bias.astype(np.int64)[None, :]
    want = np.maximum(exact, 0) + res.astype(np.int64)
    r = oracle.gemm_epilogue(A, B, "relu", bias=bias, residual=res)
    np.testing.assert_array_equal(r["out16_f64acc"], want.astype(np.float16).view(np.uint16))
    np.testing.assert_array_equal(r["out16_f32acc"], want.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("act,relu", [("relu", True), ("none", False)])
def test_plain_epilogue_matches_relu_oracle(act, relu):
    M, N, K = 30, 50, 200
    A = inputs.tensor(M, K, 12, 0)
    B = inputs.tensor(K, N, 12, 1)
    r = oracle.gemm_epilogue(A, B, act)
    p = oracle.gemm_relu(A, B, relu=relu)
    np.testing.assert_array_equal(r["out16_f64acc"], p["out16_f64acc"])
    np.testing.assert_array_equal(r["out16_f32acc"], p["out16_f32acc"])


def test_subgrid_and_argument_checks():
    M, N, K = 20, 30, 40
    A = inputs.tensor(M, K, 13, 0)
    B = inputs.tensor(K, N, 13, 1)
    bias = inputs.tensor(1, N, 14, 0).ravel()
    res = inputs.tensor(M, N, 14, 1)
    full = oracle.gemm_epilogue(A, B, "gelu_tanh", bias=bias, residual=res)
    rows, cols = np.array([19, 0, 7]), np.array([29, 3])
    sub = oracle.gemm_epilogue(A, B, "gelu_tanh", bias=bias, residual=res, rows=rows, cols=cols)
    np.testing.assert_array_equal(sub["out16_f64acc"], full["out16_f64acc"][np.ix_(rows, cols)])
    with pytest.raises(ValueError):
        oracle.gemm_epilogue(A, B, "relu", bias=bias[:-1])
    with pytest.raises(ValueError):
        oracle.gemm_epilogue(A, B, 7)


def _ulp16(y):
    return float(np.spacing(np.float16(abs(y)))) if y != 0 else 2.0 ** -24


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh"])
def test_gelu_odd_part_identity(act):
    # Both GELUs have the form x * (1 + h(x)) / 2 with h odd (erf or tanh of an odd
    # polynomial), so act(x) - act(-x) = x exactly; each output is rounded once to fp16.
    xs = np.array([0.125, 0.5, 0.75, 1.0, 1.5, 2.0, 3.0, 4.5, 7.0], np.float16)
    bias = np.concatenate([xs, -xs])
    A = np.zeros((1, 1), np.float16)
    B = np.zeros((1, bias.size), np.float16)
    out = oracle.gemm_epilogue(A, B, act, bias=bias)["out16_f64acc"].ravel().view(np.float16)
    n = xs.size
    for i, x in enumerate(xs.astype(np.float64)):
        yp, ym = float(out[i]), float(out[n + i])
        assert abs((yp - ym) - x) <= 0.5 * (_ulp16(yp) + _ulp16(ym)), (act, x, yp, ym)


def test_gelu_tanh_approximates_exact_gelu():
    # The tanh form approximates x * Phi(x) with a maximum absolute error of about 4.7e-4
    # (near |x| = 2.2); Phi comes from math.erf, independent of tanh.  A wrong cubic
    # coefficient (0.04 or 0.05 instead of 0.044715) or sqrt(pi/2) for sqrt(2/pi) exceeds the
    # 6e-4 bound where the output's fp16 spacing is fine enough to show it.
    xs = np.linspace(-6.0, 6.0, 97).astype(np.float16)
    A = np.zeros((1, 1), np.float16)
    B = np.zeros((1, xs.size), np.float16)
    out = oracle.gemm_epilogue(A, B, "gelu_tanh", bias=xs)["out16_f64acc"].ravel().view(np.float16)
    for x, y in zip(xs.astype(np.float64), out.astype(np.float64)):
        exact = x * 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))
        assert abs(y - exact) <= 6e-4 + 0.5 * _ulp16(y), (x, y, exact)


def test_gelu_limits():
    # gelu(0) = +0 or -0 (both compare equal to 0); for large x both forms return x; far left
    # they vanish (|result| below the smallest fp16 subnormal rounds to a signed zero)
    bias = np.array([0.0, 8.0, 12.0, 100.0, -30.0, -100.0], np.float16)
    A = np.zeros((1, 1), np.float16)
    B = np.zeros((1, bias.size), np.float16)
    for act in ("gelu", "gelu_tanh"):
        out = oracle.gemm_epilogue(A, B, act, bias=bias)["out16_f64acc"].ravel().view(np.float16)
        assert float(out[0]) == 0.0
        np.testing.assert_array_equal(out[1:4], bias[1:4])
        assert float(out[4]) == 0.0 and float(out[5]) == 0.0
