"""Parity of the int4-weight dequantising GEMM (tg_gemm_w4a16_f16) with the oracle:
oracle.dequant_w4 decodes the weights, oracle.gemm_epilogue multiplies; ragged M/N/K
(partial last scale group, N not a multiple of 8), both tile widths, multi-tile CTAs, the
fused epilogues and the decode-like shape on sampled outputs."""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs

from tests.parity import compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from fp16_gemm_relu_gb300 import build

    build.build()
    binding.load_library()
    torch.cuda.set_device(0)
    yield
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK, f"device error word {word:#x}"


def run_w4(a, Wq, S, N, G, act=0, bias=None, residual=None, options=None, fmt="int4"):
    M, K = a.shape
    A = torch.from_numpy(inputs.embed(a, -(-K // 8) * 8)).cuda()
    # row-major buffers whatever the caller's array layout (the ABI reads ldq / lds strides)
    Q = torch.from_numpy(np.ascontiguousarray(Wq).view(np.int32)).cuda()
    Sc = torch.from_numpy(np.ascontiguousarray(S)).cuda()
    ldc = -(-N // 8) * 8
    C = torch.full((M, ldc), float("nan"), dtype=torch.float16, device="cuda")
    b = torch.from_numpy(bias).cuda() if bias is not None else None
    r = torch.from_numpy(residual).cuda() if residual is not None else None
    fn = binding.tg_gemm_w4a16_f16 if fmt == "int4" else binding.tg_gemm_nf4a16_f16
    st = fn(A.data_ptr(), Q.data_ptr(), Sc.data_ptr(), C.data_ptr(), M, N,
                                   K, A.shape[1], Wq.shape[1], S.shape[1], ldc, G, act,
                                   b.data_ptr() if b is not None else 0,
                                   r.data_ptr() if r is not None else 0,
                                   N if r is not None else 0, options,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    out = C.cpu().numpy()
    assert np.isnan(out[:, N:]).all()
    return out[:, :N].view(np.uint16)


def make(M, N, K, G, seed, scale=None):
    a = inputs.tensor(M, K, seed, 0)
    ldq = -(-(-(-N // 8)) // 4) * 4
    Wq = inputs.int4_weights(K, N, seed, ldq=ldq)
    S = inputs.int4_scales(-(-K // G), N, seed, scale or 1.0 / np.sqrt(K), lds=-(-N // 8) * 8)
    return a, Wq, S


def check(got, a, Wq, S, N, G, act="none", bias=None, residual=None, rows=None, cols=None,
          fmt="int4"):
    K = a.shape[1]
    w = (oracle.dequant_w4 if fmt == "int4" else oracle.dequant_nf4)(Wq, S, K, N, G)
    r = oracle.gemm_epilogue(a, w, act, bias=bias, residual=residual, rows=rows, cols=cols)
    ref = {"out16_f64acc": r["out16_f64acc"], "acc_f64": r["pre_f64"]}
    zr = act == "relu" and residual is None
    c = compare(got, ref, K, relu=zr)
    assert c["out_of_tol"] == 0 and (not zr or c["zero_rule"] == 0), c
    return c


@pytest.mark.parametrize("M,N,K,G", [(128, 256, 128, 64), (333, 527, 1030, 128),
                                     (64, 1000, 4096, 128), (700, 300, 640, 256)])
@pytest.mark.parametrize("bn", [128, 256])
def test_w4_parity(M, N, K, G, bn):
    a, Wq, S = make(M, N, K, G, 7)
    got = run_w4(a, Wq, S, N, G, options={"block_n": bn})
    check(got, a, Wq, S, N, G)


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_w4_epilogue_and_multitile(act):
    M, N, K, G = 400, 600, 1024, 128
    a, Wq, S = make(M, N, K, G, 8)
    bias = inputs.tensor(1, N, 9, 0).ravel()
    res = inputs.tensor(M, N, 9, 1)
    ACT = {"relu": 1, "gelu": 2}
    got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res,
                 options={"max_ctas": 3, "block_n": 128})
    check(got, a, Wq, S, N, G, act, bias, res)
    got0 = run_w4(a, Wq, S, N, G, act=ACT[act], options={"max_ctas": 2})
    check(got0, a, Wq, S, N, G, act)


@pytest.mark.parametrize("M,N,K,G", [(1, 257, 640, 128), (64, 1000, 4096, 128), (100, 300, 1030, 64),
                                     (128, 2048, 2048, 256), (37, 520, 1000, 192)])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_w4_swapped_kernel(M, N, K, G, act):
    # C^T = W^T A^T with the decoded weights on the MMA's 128-row side (small M)
    a, Wq, S = make(M, N, K, G, 11)
    ACT = {"none": 0, "relu": 1, "gelu": 2}
    bias = inputs.tensor(1, N, 12, 0).ravel()
    res = inputs.tensor(M, N, 12, 1)
    got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res, options={"swap_ab": 1})
    check(got, a, Wq, S, N, G, act, bias, res)
    got0 = run_w4(a, Wq, S, N, G, act=ACT[act], options={"swap_ab": 1, "max_ctas": 3})
    check(got0, a, Wq, S, N, G, act)


def test_w4_decode_shape_sampled():
    M, N, K, G = 64, 28672, 8192, 128
    a = inputs.tensor(M, K, 3, 0, "normal")
    Wq = inputs.int4_weights(K, N, 3)
    S = inputs.int4_scales(K // G, N, 3, 1.0 / np.sqrt(K))
    got = run_w4(a, Wq, S, N, G, act=1)
    rng = np.random.default_rng(0)
    cols = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 200)]))
    rows = np.arange(M)
    check(got[np.ix_(rows, cols)], a, Wq[:, :], S, N, G, "relu", rows=rows, cols=cols)


def test_w4_square_workload_sampled():
    # the int4 bench workload at full size: square8192's A, weights and scales as the bench
    # makes them, sampled rows and columns across tile and cluster boundaries, in the default
    # launch (decode first, then the fp16 GEMM) and with the fused CTA-pair kernel
    from fp16_gemm_relu_gb300 import workloads

    wl = workloads.get("square8192")
    M, N, K, G = wl.M, wl.N, wl.K, 128
    a = wl.make_a()
    Wq = inputs.int4_weights(K, N, wl.seed)
    S = inputs.int4_scales(K // G, N, wl.seed, 1.0 / np.sqrt(K))
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], rng.integers(0, M, 40)]))
    cols = np.unique(np.concatenate([[0, 7, 8, 127, 128, 255, 256, N - 1],
                                     rng.integers(0, N, 40)]))
    for opts in (None, {"pair": 1}):
        got = run_w4(a, Wq, S, N, G, act=1, options=opts)
        check(got[np.ix_(rows, cols)], a, Wq, S, N, G, "relu", rows=rows, cols=cols)


@pytest.mark.parametrize("fmt", ["int4", "nf4"])
@pytest.mark.parametrize("M,N,K,G", [(1, 257, 640, 128), (300, 527, 1030, 128), (800, 1000, 640, 192),
                                     (129, 1301, 1537, 64)])
@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_decode_first(fmt, M, N, K, G, act):
    # the whole weight matrix decoded to fp16 scratch, then the fp16 GEMM: ragged N (the last
    # packed word's columns past N), partial scale groups, fused epilogues
    a, Wq, S = make(M, N, K, G, 41)
    ACT = {"relu": 1, "gelu_tanh": 3}
    bias = inputs.tensor(1, N, 42, 0).ravel()
    res = inputs.tensor(M, N, 42, 1)
    got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res,
                 options={"dequant_first": 1}, fmt=fmt)
    check(got, a, Wq, S, N, G, act, bias, res, fmt=fmt)
    got0 = run_w4(a, Wq, S, N, G, act=1, options={"dequant_first": 1, "max_ctas": 3}, fmt=fmt)
    check(got0, a, Wq, S, N, G, "relu", fmt=fmt)


@pytest.mark.parametrize("fmt", ["int4", "nf4"])
def test_decode_first_is_the_default_for_large_m(fmt):
    # with no kernel override, a large M takes the decode-first plan: bitwise what forcing it
    # gives (each plan is deterministic)
    M, N, K, G = 1024, 768, 2048, 128
    a, Wq, S = make(M, N, K, G, 43)
    auto = run_w4(a, Wq, S, N, G, act=1, fmt=fmt)
    forced = run_w4(a, Wq, S, N, G, act=1, options={"dequant_first": 1}, fmt=fmt)
    np.testing.assert_array_equal(auto, forced)
    check(auto, a, Wq, S, N, G, "relu", fmt=fmt)
    fused = run_w4(a, Wq, S, N, G, act=1, options={"dequant_first": -1}, fmt=fmt)
    check(fused, a, Wq, S, N, G, "relu", fmt=fmt)


@pytest.mark.parametrize("fmt,M,first", [("int4", 511, False), ("int4", 512, True),
                                          ("nf4", 383, False), ("nf4", 384, True)])
def test_decode_first_threshold(fmt, M, first):
    # the default switches to decode-first at M = 512 for int4 and M = 384 for NF4 weights
    # (NF4's fused decode costs more): bitwise what forcing that plan gives, and the oracle's
    N, K, G = 520, 1030, 128
    a, Wq, S = make(M, N, K, G, 44)
    auto = run_w4(a, Wq, S, N, G, act=1, fmt=fmt)
    forced = run_w4(a, Wq, S, N, G, act=1, options={"dequant_first": 1 if first else -1},
                    fmt=fmt)
    np.testing.assert_array_equal(auto, forced)
    check(auto, a, Wq, S, N, G, "relu", fmt=fmt)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_w4_swapped_small_grid_ragged_fused_epilogue(act):
    # several tiles per CTA (2 and 3 CTAs for 6 column tiles), a ragged last tile (N = 700
    # leaves a partial warp of columns), M = 90 under a 128-row tile, bias + residual + the
    # activation, repeated: the epilogue of one tile overlaps the next tile's main loop
    M, N, K, G = 90, 700, 1536, 128
    a, Wq, S = make(M, N, K, G, 22)
    ACT = {"relu": 1, "gelu_tanh": 3}
    bias = inputs.tensor(1, N, 23, 0).ravel()
    res = inputs.tensor(M, N, 23, 1)
    first = {}
    for rep in range(4):
        for cap in (2, 3):
            got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res,
                         options={"swap_ab": 1, "max_ctas": cap})
            if rep == 0:
                check(got, a, Wq, S, N, G, act, bias, res)
                first[cap] = got
            else:  # the plan fixes the summation order: repeated calls are bitwise equal
                np.testing.assert_array_equal(got, first[cap])


@pytest.mark.parametrize("cap,tail", [(4, 1), (4, 0), (8, 0), (8, -1), (3, 1)])
def test_w4_swapped_tail_split(cap, tail):
    # 11 column tiles: with 4 CTAs the last wave holds 3 tiles (split only when forced), with 8
    # CTAs it holds 3 of 8 (split by default: 6 half-tiles fit one wave), with 3 CTAs 2 of 3.
    # K = 1030 gives 17 k-blocks: halves of 9 and 8, the second ending in a partial block and a
    # partial scale group.  Split tiles meet through the float32 workspace; the result must
    # match the oracle and repeat bit for bit (a + b == b + a, whichever half lands second).
    M, N, K, G = 90, 1300, 1030, 64
    a, Wq, S = make(M, N, K, G, 31)
    bias = inputs.tensor(1, N, 32, 0).ravel()
    res = inputs.tensor(M, N, 32, 1)
    opts = {"swap_ab": 1, "max_ctas": cap, "tail": tail}
    got = run_w4(a, Wq, S, N, G, act=3, bias=bias, residual=res, options=opts)
    check(got, a, Wq, S, N, G, "gelu_tanh", bias, res)
    for _ in range(3):
        np.testing.assert_array_equal(run_w4(a, Wq, S, N, G, act=3, bias=bias, residual=res,
                                             options=opts), got)
    plain = run_w4(a, Wq, S, N, G, act=1, options=opts)
    check(plain, a, Wq, S, N, G, "relu")


def test_w4_swapped_tail_split_single_k_block():
    # one k-block cannot be halved: the forced split falls back to whole tiles
    M, N, K, G = 64, 1300, 64, 64
    a, Wq, S = make(M, N, K, G, 33)
    got = run_w4(a, Wq, S, N, G, act=1, options={"swap_ab": 1, "max_ctas": 4, "tail": 1})
    check(got, a, Wq, S, N, G, "relu")


@pytest.mark.parametrize("M,N,K,G", [(256, 256, 128, 64), (333, 527, 1030, 128), (700, 1000, 640, 256),
                                     (1024, 768, 2048, 128), (300, 600, 1000, 192)])
def test_w4_pair_kernel(M, N, K, G):
    # 256 x 256 tiles on CTA pairs, each CTA decoding its 128 columns; ragged M / N / K
    a, Wq, S = make(M, N, K, G, 31)
    got = run_w4(a, Wq, S, N, G, options={"pair": 1})
    check(got, a, Wq, S, N, G)
    got1 = run_w4(a, Wq, S, N, G, options={"pair": 1, "max_ctas": 2})  # one cluster, all tiles
    check(got1, a, Wq, S, N, G)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_w4_pair_fused_epilogue(act):
    M, N, K, G = 520, 700, 1536, 128
    a, Wq, S = make(M, N, K, G, 32)
    ACT = {"relu": 1, "gelu_tanh": 3}
    bias = inputs.tensor(1, N, 33, 0).ravel()
    res = inputs.tensor(M, N, 33, 1)
    got = run_w4(a, Wq, S, N, G, act=ACT[act], bias=bias, residual=res,
                 options={"pair": 1, "max_ctas": 4})
    check(got, a, Wq, S, N, G, act, bias, res)


@pytest.mark.parametrize("fmt", ["int4", "nf4"])
@pytest.mark.parametrize("M,N,K,G", [(1, 257, 640, 128), (37, 1300, 1030, 64), (64, 2048, 4096, 128),
                                     (64, 520, 64, 64)])
def test_tmem_decode_matches_shared_memory_decode(fmt, M, N, K, G):
    # on request, with at most 64 rows of A, the swapped kernel decodes the weights into
    # tensor memory and the MMA reads them there; the same weights in the same K order through
    # shared memory must give the same bits, and both match the oracle (default grid with the
    # split tail, and a small grid with several tiles per CTA)
    a, Wq, S = make(M, N, K, G, 51)
    bias = inputs.tensor(1, N, 52, 0).ravel()
    for extra in ({}, {"max_ctas": 3}):
        t = run_w4(a, Wq, S, N, G, act=1, bias=bias,
                   options={"swap_ab": 1, "tmem_decode": 1, **extra}, fmt=fmt)
        sm = run_w4(a, Wq, S, N, G, act=1, bias=bias, options={"swap_ab": 1, **extra}, fmt=fmt)
        np.testing.assert_array_equal(t, sm)
        check(t, a, Wq, S, N, G, "relu", bias, fmt=fmt)
