"""Pins for the oracle's int4 weight decoding, w = fp16_rne((q - 8) * s): an independent numpy
unpacking and rounding, and hand-picked closed forms (zero point, exact scales, overflow)."""

import numpy as np

import oracle
from fp16_gemm_relu_gb300 import inputs


def _numpy_dequant(Wq, S, K, N, G):
    n = np.arange(N)
    q = (Wq[:, n // 8] >> (4 * (n % 8)).astype(np.uint32)) & 0xF
    s = S[np.arange(K) // G][:, :N].astype(np.float64)
    with np.errstate(over="ignore"):
        return ((q.astype(np.float64) - 8.0) * s).astype(np.float16)


def test_against_numpy_unpacking():
    K, N, G = 300, 77, 128
    Wq = inputs.int4_weights(K, N, 5, ldq=12)
    S = inputs.int4_scales((K + G - 1) // G, N, 5, 0.02, lds=80)
    got = oracle.dequant_w4(Wq, S, K, N, G)
    np.testing.assert_array_equal(got.view(np.uint16), _numpy_dequant(Wq, S, K, N, G).view(np.uint16))


def test_closed_forms():
    # one row, eight columns: nibbles 0..7 then 8..15 in the second word
    Wq = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    ones = np.ones((1, 16), np.float16)
    np.testing.assert_array_equal(oracle.dequant_w4(Wq, ones, 1, 16, 64)[0].astype(np.float64),
                                  np.arange(16) - 8.0)
    # power-of-two scale: exact; zero point gives +0 for a positive scale
    quarter = np.full((1, 16), 0.25, np.float16)
    w = oracle.dequant_w4(Wq, quarter, 1, 16, 64)
    np.testing.assert_array_equal(w[0].astype(np.float64), (np.arange(16) - 8.0) * 0.25)
    assert w.view(np.uint16)[0, 8] == 0x0000
    # (0 - 8) * 65504 overflows to -inf; 7 * 65504 to +inf; 3 * 1.0009765625 rounds to even
    big = np.full((1, 16), 65504.0, np.float16)
    wb = oracle.dequant_w4(Wq, big, 1, 16, 64)
    assert np.isneginf(wb[0, 0]) and np.isposinf(wb[0, 15]) and wb[0, 9] == np.float16(65504.0)
    odd = np.full((1, 16), 1.0009765625, np.float16)  # 1 + 2^-10
    wo = oracle.dequant_w4(Wq, odd, 1, 16, 64)
    # 3 * (1 + 2^-10) = 3 + 3*2^-10 lies between fp16 neighbours 3 + 2^-9 and 3 + 2^-8 (spacing
    # 2^-9 in [2, 4)): it is 3 + 1.5*2^-9, a tie, which goes to the even one, 3 + 2^-8
    assert wo[0, 11] == np.float16(3.00390625)


def test_group_boundaries():
    K, N, G = 256, 16, 64
    Wq = np.tile(np.array([[0x99999999, 0x99999999]], np.uint32), (K, 1))  # q = 9 -> 1 * s
    S = np.arange(1, 5, dtype=np.float16)[:, None].repeat(16, axis=1)       # group g -> g + 1
    w = oracle.dequant_w4(Wq, S, K, N, G)
    np.testing.assert_array_equal(w[:, 0].astype(np.float64), (np.arange(K) // G) + 1.0)
