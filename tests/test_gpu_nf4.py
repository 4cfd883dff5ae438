"""Parity of the NF4-weight dequantising GEMM (tg_gemm_nf4a16_f16, the W_NF4 / A_FP16 case of
the TileLang paper-reading page, section 5) with the oracle: oracle.dequant_nf4 decodes the
weights with QLoRA's code table, oracle.gemm_epilogue multiplies.  Every code value, all three
kernels (swapped-operand, single-CTA, CTA pair), ragged M / N / K, partial scale groups,
fused epilogues, the swapped kernel's split tail, and the decode-like shape on sampled
outputs."""

import numpy as np
import pytest

from fp16_gemm_relu_gb300 import binding, inputs

from tests.test_gpu_w4 import _built, check, make, run_w4  # noqa: F401

pytestmark = pytest.mark.gpu


def test_nf4_every_code_value():
    # A = identity rows: C = W exactly (one product per output, K = 64 rows of weights), with
    # words that hold every code 0..15 in every nibble position
    K, N, G = 64, 128, 64
    a = np.zeros((K, K), np.float16)
    np.fill_diagonal(a, 1.0)
    base = np.array([0x76543210, 0xFEDCBA98, 0x13579BDF, 0x02468ACE], np.uint32)
    Wq = np.ascontiguousarray(np.stack([np.roll(base, r) for r in range(K)])[:, np.arange(16) % 4])
    S = inputs.int4_scales(1, N, 5, 0.5, lds=N)
    for opts in ({"swap_ab": 1}, {"swap_ab": -1, "block_n": 128}, {"swap_ab": -1, "pair": 1},
                 {"dequant_first": 1}):
        got = run_w4(a, Wq, S, N, G, options=opts, fmt="nf4")
        check(got, a, Wq, S, N, G, fmt="nf4")


@pytest.mark.parametrize("M,N,K,G", [(128, 256, 128, 64), (333, 527, 1030, 128),
                                     (700, 300, 640, 256)])
@pytest.mark.parametrize("bn", [128, 256])
def test_nf4_single_cta_kernel(M, N, K, G, bn):
    a, Wq, S = make(M, N, K, G, 17)
    got = run_w4(a, Wq, S, N, G, options={"swap_ab": -1, "block_n": bn}, fmt="nf4")
    check(got, a, Wq, S, N, G, fmt="nf4")


@pytest.mark.parametrize("M,N,K,G", [(1, 257, 640, 128), (64, 1000, 4096, 128),
                                     (100, 300, 1030, 64), (37, 520, 1000, 192)])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_nf4_swapped_kernel(M, N, K, G, act):
    a, Wq, S = make(M, N, K, G, 18)
    ACT = {"none": 0, "relu": 1, "gelu": 2}
    bias = inputs.tensor(1, N, 19, 0).ravel()
    res = inputs.tensor(M, N, 19, 1)
    got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res, options={"swap_ab": 1},
                 fmt="nf4")
    check(got, a, Wq, S, N, G, act, bias, res, fmt="nf4")
    got0 = run_w4(a, Wq, S, N, G, act=ACT[act], options={"swap_ab": 1, "max_ctas": 3},
                  fmt="nf4")
    check(got0, a, Wq, S, N, G, act, fmt="nf4")


@pytest.mark.parametrize("M,N,K,G", [(256, 256, 128, 64), (333, 527, 1030, 128),
                                     (1024, 768, 2048, 128), (300, 600, 1000, 192)])
def test_nf4_pair_kernel(M, N, K, G):
    a, Wq, S = make(M, N, K, G, 20)
    got = run_w4(a, Wq, S, N, G, options={"pair": 1}, fmt="nf4")
    check(got, a, Wq, S, N, G, fmt="nf4")
    got1 = run_w4(a, Wq, S, N, G, options={"pair": 1, "max_ctas": 2}, fmt="nf4")
    check(got1, a, Wq, S, N, G, fmt="nf4")


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_nf4_fused_epilogues(act):
    M, N, K, G = 520, 700, 1536, 128
    a, Wq, S = make(M, N, K, G, 21)
    ACT = {"relu": 1, "gelu_tanh": 3}
    bias = inputs.tensor(1, N, 22, 0).ravel()
    res = inputs.tensor(M, N, 22, 1)
    for opts in ({"pair": 1, "max_ctas": 4}, {"block_n": 256, "max_ctas": 3}):
        got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res, options=opts,
                     fmt="nf4")
        check(got, a, Wq, S, N, G, act, bias, res, fmt="nf4")


@pytest.mark.parametrize("cap,tail", [(4, 1), (8, 0)])
def test_nf4_swapped_tail_split(cap, tail):
    M, N, K, G = 90, 1300, 1030, 64
    a, Wq, S = make(M, N, K, G, 23)
    opts = {"swap_ab": 1, "max_ctas": cap, "tail": tail}
    got = run_w4(a, Wq, S, N, G, act=1, options=opts, fmt="nf4")
    check(got, a, Wq, S, N, G, "relu", fmt="nf4")
    for _ in range(2):
        np.testing.assert_array_equal(run_w4(a, Wq, S, N, G, act=1, options=opts, fmt="nf4"),
                                      got)


def test_nf4_decode_shape_sampled():
    M, N, K, G = 64, 28672, 8192, 128
    a = inputs.tensor(M, K, 3, 0, "normal")
    Wq = inputs.int4_weights(K, N, 3)
    S = inputs.int4_scales(K // G, N, 3, 1.0 / np.sqrt(K))
    got = run_w4(a, Wq, S, N, G, act=1, fmt="nf4")
    rng = np.random.default_rng(2)
    cols = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 200)]))
    rows = np.arange(M)
    check(got[np.ix_(rows, cols)], a, Wq, S, N, G, "relu", rows=rows, cols=cols, fmt="nf4")


def test_nf4_argument_errors_match_int4():
    p = 4096
    for fn in (binding.tg_gemm_w4a16_f16, binding.tg_gemm_nf4a16_f16):
        assert fn(p, p, p, p, 4, 4, 64, 64, 4, 8, 8, 32) == binding.TG_ERR_INVALID_ARG
        assert fn(p + 2, p, p, p, 4, 8, 64, 64, 4, 8, 8, 64) == binding.TG_ERR_MISALIGNED
