"""Pins for the oracle's backward of relu(A·B): the mask on hand-picked special values, and
the whole backward against torch's float64 autograd on CPU (an independent implementation:
the oracle's sums are its own C loops)."""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import inputs

from tests.parity import compare

torch = pytest.importorskip("torch")


def test_relu_backward_special_values():
    C = np.array([1.0, 0.0, -0.0, -1.0, np.nan, np.inf, 2.0 ** -24, -np.inf], np.float16)
    dC = np.array([3.0, 5.0, -7.0, 9.0, 11.0, -13.0, 0.5, 2.0], np.float16)
    got = oracle.relu_backward(dC, C)
    want = np.array([3.0, 0.0, 0.0, 0.0, 0.0, -13.0, 0.5, 0.0], np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)
    assert not (got == 0x8000).any()  # masked entries are +0 even where dC < 0


@pytest.mark.parametrize("M,N,K", [(17, 23, 31), (64, 40, 96)])
def test_backward_matches_float64_autograd(M, N, K):
    a = inputs.tensor(M, K, 200 + M, 0)
    b = inputs.tensor(K, N, 200 + M, 1)
    c = oracle.f16_bits_to_f64(oracle.gemm_relu(a, b)["out16_f64acc"]).astype(np.float16)
    dc = inputs.tensor(M, N, 300 + M, 1)
    got = oracle.relu_matmul_backward(a, b, c, dc)
    # float64 autograd through relu, masked on the fp16 forward output like the definition
    A = torch.tensor(a.astype(np.float64), requires_grad=True)
    B = torch.tensor(b.astype(np.float64), requires_grad=True)
    Z = A @ B
    mask = torch.tensor(c.astype(np.float64) > 0)
    (Z * mask).backward(torch.tensor(dc.astype(np.float64)))
    dz = np.where(c > 0, dc, np.float16(0))
    np.testing.assert_array_equal(got["dZ"], dz.view(np.uint16))
    for key, g, Kred in (("dA", A.grad, N), ("dB", B.grad, M)):
        ref = {"out16_f64acc": g.numpy().astype(np.float16).view(np.uint16),
               "acc_f64": g.numpy()}
        c_ = compare(got[key]["out16_f64acc"], ref, Kred, relu=False)
        assert c_["out_of_tol"] == 0 and c_["max_ulp_err"] <= 1.0, (key, c_)
