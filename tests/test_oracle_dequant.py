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


# ---- NF4 (QLoRA's 4-bit NormalFloat, the W_NF4 / A_FP16 case of the paper-reading page,
# section 5) ----

def _nf4_construction():
    """NF4 rebuilt from its definition (QLoRA, section 3): quantiles of a standard normal taken
    separately for the two signs so that 0 is a code: 8 positive quantiles at probabilities
    evenly spaced from delta down to (not including) 1/2, 7 negative ones the same way with 7
    steps, and 0; all divided by the largest, so the codes span [-1, 1].  delta, the outermost
    probability, is the mean of 1 - 1/(2*15) and 1 - 1/(2*16)."""
    stats = __import__("pytest").importorskip("scipy.stats")
    d = 0.5 * ((1 - 1 / 30) + (1 - 1 / 32))
    pos = [stats.norm.ppf(d - j * (d - 0.5) / 8) for j in range(8)]
    neg = [-stats.norm.ppf(d - j * (d - 0.5) / 7) for j in range(7)]
    return np.sort(np.array(pos + [0.0] + neg)) / stats.norm.ppf(d)


def test_nf4_table_structure():
    c = oracle.nf4_codes()
    assert c.shape == (16,)
    assert (np.diff(c) > 0).all()
    assert c[0] == -1.0 and c[15] == 1.0 and c[7] == 0.0
    assert (c[:7] < 0).all() and (c[8:] > 0).all()


def test_nf4_table_matches_the_quantile_construction():
    c = oracle.nf4_codes()
    v = _nf4_construction()
    # the printed table was computed in float32: agreement to a few float32 ulps
    assert np.max(np.abs(c - v)) < 1e-6, np.abs(c - v)
    # and, what the decode uses, both round to the same fp16 codes
    np.testing.assert_array_equal(c.astype(np.float16).view(np.uint16),
                                  v.astype(np.float16).view(np.uint16))


def _numpy_dequant_nf4(Wq, S, K, N, G):
    n = np.arange(N)
    q = (Wq[:, n // 8] >> (4 * (n % 8)).astype(np.uint32)) & 0xF
    code16 = _nf4_construction().astype(np.float16).astype(np.float64)
    s = S[np.arange(K) // G][:, :N].astype(np.float64)
    with np.errstate(over="ignore"):
        return (code16[q] * s).astype(np.float16)


def test_nf4_against_numpy_unpacking():
    K, N, G = 300, 77, 128
    Wq = inputs.int4_weights(K, N, 6, ldq=12)
    S = inputs.int4_scales((K + G - 1) // G, N, 6, 0.02, lds=80)
    got = oracle.dequant_nf4(Wq, S, K, N, G)
    np.testing.assert_array_equal(got.view(np.uint16),
                                  _numpy_dequant_nf4(Wq, S, K, N, G).view(np.uint16))


def test_nf4_closed_forms():
    Wq = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)  # codes 0..15 in order
    ones = np.ones((1, 16), np.float16)
    w = oracle.dequant_nf4(Wq, ones, 1, 16, 64)[0]
    assert w[0] == -1.0 and w[15] == 1.0 and w.view(np.uint16)[7] == 0x0000
    # code 13 is 0.5626170...: in fp16 (spacing 2^-11 in [0.5, 1)) it is 0.5625 = 9/16
    assert w[13] == np.float16(0.5625)
    # scale 1 + 4 * 2^-10: 9/16 * (1 + 2^-8) = 9/16 + 4.5 * 2^-11, a tie between mantissas
    # 128 + 4 and 128 + 5 that goes to the even one: 0x3884.  Rounding the code value's full
    # precision instead (0.5626170 * 1.00390625 = 0.5648148) would give 0x3885.
    tie = np.full((1, 16), 1.00390625, np.float16)
    assert oracle.dequant_nf4(Wq, tie, 1, 16, 64).view(np.uint16)[0, 13] == 0x3884
    # a power-of-two scale is exact; the zero code times a negative scale is -0
    neg = np.full((1, 16), -0.25, np.float16)
    wn = oracle.dequant_nf4(Wq, neg, 1, 16, 64)
    np.testing.assert_array_equal(wn[0].astype(np.float64), -0.25 * w.astype(np.float64))
    assert wn.view(np.uint16)[0, 7] == 0x8000
    # group boundaries: scale row g applies to rows [g G, (g + 1) G)
    K, N, G = 256, 16, 64
    Wq2 = np.tile(np.array([[0xFFFFFFFF, 0xFFFFFFFF]], np.uint32), (K, 1))  # code 1.0
    S2 = np.arange(1, 5, dtype=np.float16)[:, None].repeat(16, axis=1)
    np.testing.assert_array_equal(oracle.dequant_nf4(Wq2, S2, K, N, G)[:, 3].astype(np.float64),
                                  (np.arange(K) // G) + 1.0)
