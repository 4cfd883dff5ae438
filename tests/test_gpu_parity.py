"""Parity of the CUDA path (through the C ABI) with the oracle, element by element, on seeded
inputs: every tile width, split-K on and off, repacked operands, the workspace epilogue,
multi-tile-per-CTA schedules, ragged tails, odd leading dimensions and pointers, empty and
degenerate shapes, and the integer-input case where any summation order is exact."""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs

from tests.parity import assert_parity

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


def _dev(x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_gpu(a, b, relu=True, options=None, lda=None, ldb=None, ldc=None, a_off=0, b_off=0,
            c_off=0, fill=np.nan):
    """Run through tg_gemm_relu_f16(_ex) with optional padded leading dimensions and element
    offsets of the base pointers (odd offsets give 2-byte-aligned pointers).  Returns the C
    bits (M, N) and the untouched-canary check of the padding."""
    M, K = a.shape
    N = b.shape[1]
    lda = lda or max(K, 1)
    ldb = ldb or max(N, 1)
    ldc = ldc or max(N, 1)
    abuf = np.full(a_off + M * lda + 8, fill, dtype=np.float16)
    abuf[a_off:a_off + M * lda].reshape(M, lda)[:, :K] = a
    bbuf = np.full(b_off + K * ldb + 8, fill, dtype=np.float16)
    bbuf[b_off:b_off + K * ldb].reshape(K, ldb)[:, :N] = b
    canary = np.uint16(0x7E5A)
    cbuf = np.full(c_off + M * ldc + 8, canary, dtype=np.uint16)
    dA, dB, dC = _dev(abuf), _dev(bbuf), _dev(cbuf)
    pa = dA.data_ptr() + 2 * a_off
    pb = dB.data_ptr() + 2 * b_off
    pc = dC.data_ptr() + 2 * c_off
    flag = binding.TG_EPILOGUE_RELU if relu else binding.TG_EPILOGUE_NONE
    stream = torch.cuda.current_stream().cuda_stream
    if options is None:
        st = binding.tg_gemm_relu_f16(pa, pb, pc, M, N, K, lda, ldb, ldc, flag, stream)
    else:
        st = binding.tg_gemm_relu_f16_ex(pa, pb, pc, M, N, K, lda, ldb, ldc, flag, options, stream)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    c = out[c_off:c_off + M * ldc].reshape(M, ldc)
    pad_ok = bool((c[:, N:] == canary).all() and (out[:c_off] == canary).all()
                  and (out[c_off + M * ldc:] == canary).all())
    return np.ascontiguousarray(c[:, :N]), pad_ok


def oracle_ref(a, b, relu=True, rows=None, cols=None):
    return oracle.gemm_relu(a, b, relu=relu, rows=rows, cols=cols)


SHAPES = [(1, 1, 1), (7, 13, 5), (128, 256, 64), (129, 257, 65), (255, 300, 1000),
          (300, 520, 777), (64, 1000, 3000), (1000, 777, 1031)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("relu", [True, False])
def test_default_plan_parity(M, N, K, relu):
    a = inputs.tensor(M, K, 1000 + M, 0)
    b = inputs.tensor(K, N, 1000 + M, 1)
    c, pad_ok = run_gpu(a, b, relu)
    assert pad_ok
    assert_parity(c, oracle_ref(a, b, relu), K, relu, where=f"{M}x{N}x{K}")


FORCED = [
    {"block_n": 256}, {"block_n": 192}, {"block_n": 128},
    {"split_k": 2}, {"split_k": 3, "block_n": 192}, {"split_k": 7, "block_n": 128},
    {"force_repack": 1}, {"force_workspace": 1},
    {"max_ctas": 1}, {"max_ctas": 3, "split_k": 2}, {"max_ctas": 5, "panel_m": 1},
    {"max_ctas": 2, "block_n": 128, "panel_m": 2},
    {"pair": 1}, {"pair": 1, "split_k": 3}, {"pair": 1, "max_ctas": 2},
    {"pair": 1, "max_ctas": 6, "panel_m": 1}, {"pair": 1, "force_repack": 1},
    {"pair": 1, "force_workspace": 1}, {"pair": -1},
    {"pair": 1, "tail": 1, "max_ctas": 8}, {"pair": 1, "tail": 1, "max_ctas": 10},
]


@pytest.mark.parametrize("opts", FORCED, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_forced_plans_parity(opts):
    M, N, K = 300, 600, 1500
    a = inputs.tensor(M, K, 77, 0)
    b = inputs.tensor(K, N, 77, 1)
    c, pad_ok = run_gpu(a, b, True, options=opts)
    assert pad_ok
    assert_parity(c, oracle_ref(a, b, True), K, True, where=str(opts))


@pytest.mark.parametrize("opts", [None, {"split_k": 4}, {"max_ctas": 3},
                                  {"force_repack": 1, "split_k": 3}, {"pair": 1},
                                  {"pair": 1, "split_k": 5, "max_ctas": 4},
                                  {"pair": 1, "tail": 1, "max_ctas": 8}])
@pytest.mark.parametrize("M,N,K", [(200, 300, 700), (129, 65, 4099)])
def test_integer_inputs_bitwise(opts, M, N, K):
    a = inputs.tensor(M, K, 5, 0, "int")
    b = inputs.tensor(K, N, 5, 1, "int")
    for relu in (True, False):
        c, _ = run_gpu(a, b, relu, options=opts)
        np.testing.assert_array_equal(c.view(np.uint16),
                                      oracle_ref(a, b, relu)["out16_f32acc"])


@pytest.mark.parametrize("case", [
    dict(lda=1037, ldb=531, ldc=531),             # odd leading dimensions
    dict(lda=1040, ldb=536, ldc=536),             # padded, 16-byte aligned
    dict(a_off=1, b_off=3, c_off=5),              # 2-byte-aligned pointers
    dict(lda=1033, ldb=529, ldc=533, a_off=7, b_off=1, c_off=1),
])
@pytest.mark.parametrize("pair", [-1, 1])
def test_strides_and_pointer_offsets(case, pair):
    M, N, K = 333, 527, 1030
    a = inputs.tensor(M, K, 9, 0)
    b = inputs.tensor(K, N, 9, 1)
    c, pad_ok = run_gpu(a, b, True, options={"pair": pair}, **case)
    assert pad_ok, "wrote outside the M x N region of C"
    assert_parity(c, oracle_ref(a, b, True), K, True, where=f"{case} pair={pair}")


def test_k_zero_writes_positive_zero():
    M, N = 37, 45
    a = np.zeros((M, 0), np.float16)
    b = np.zeros((0, N), np.float16)
    c, pad_ok = run_gpu(a, b, True, lda=1, ldb=N)
    assert pad_ok and (c.view(np.uint16) == 0).all()
    c, _ = run_gpu(a, b, False, lda=1, ldb=N)
    assert (c.view(np.uint16) == 0).all()


def test_empty_outputs_are_noops():
    for M, N, K in [(0, 5, 5), (5, 0, 5), (0, 0, 0)]:
        st = binding.tg_gemm_relu_f16(0, 0, 0, M, N, K, max(K, 1), max(N, 1), max(N, 1), 1, 0)
        assert st == binding.TG_OK


def test_all_negative_products_are_exact_zero():
    M, N, K = 257, 383, 2000
    a = np.abs(inputs.tensor(M, K, 13, 0)) + np.float16(0.01)
    b = -(np.abs(inputs.tensor(K, N, 13, 1)) + np.float16(0.01))
    for opts in (None, {"split_k": 3}):
        c, _ = run_gpu(a, b, True, options=opts)
        assert (c.view(np.uint16) == 0).all()
        c0, _ = run_gpu(a, b, False, options=opts)
        assert (c0.view(np.uint16) & 0x8000).all()


def test_relu_of_identity_epilogue_and_determinism():
    M, N, K = 400, 700, 3000
    a = inputs.tensor(M, K, 17, 0)
    b = inputs.tensor(K, N, 17, 1)
    for opts in (None, {"split_k": 5}, {"block_n": 128, "max_ctas": 7}, {"pair": 1},
                 {"pair": 1, "split_k": 3, "max_ctas": 4}, {"pair": 1, "tail": 1, "max_ctas": 6}):
        c1, _ = run_gpu(a, b, True, options=opts)
        c2, _ = run_gpu(a, b, True, options=opts)
        np.testing.assert_array_equal(c1.view(np.uint16), c2.view(np.uint16))
        c0, _ = run_gpu(a, b, False, options=opts)
        bits = c0.view(np.uint16)
        np.testing.assert_array_equal(c1.view(np.uint16), np.where(bits & 0x8000, 0, bits))


def test_split_k_agrees_with_single_pass():
    M, N, K = 256, 512, 8192
    a = inputs.tensor(M, K, 23, 0)
    b = inputs.tensor(K, N, 23, 1)
    ref = oracle_ref(a, b, True)
    for s in (1, 2, 4, 16):
        for pair in (-1, 1):
            c, _ = run_gpu(a, b, True, options={"split_k": s, "pair": pair})
            assert_parity(c, ref, K, True, where=f"split_k={s} pair={pair}")


def test_permutation_is_exact():
    n, N = 300, 700
    perm = np.random.default_rng(3).permutation(n)
    P = np.zeros((n, n), np.float16)
    P[np.arange(n), perm] = 1
    b = inputs.tensor(n, N, 29, 1)
    c, _ = run_gpu(P, b, False)
    np.testing.assert_array_equal(c.view(np.uint16), b[perm].view(np.uint16))


def test_subnormal_inputs_are_not_flushed():
    # products of fp16 subnormals and ones: exact sums in the subnormal range
    M, N, K = 130, 260, 70
    a = np.full((M, K), np.float16(2.0 ** -24))
    a[:, 1::2] = np.float16(3 * 2.0 ** -24)
    b = np.ones((K, N), np.float16)
    c, _ = run_gpu(a, b, True)
    want = oracle_ref(a, b, True)["out16_f32acc"]
    np.testing.assert_array_equal(c.view(np.uint16), want)
    assert (want != 0).all()


def test_host_buffer_entry_point():
    M, N, K = 300, 517, 999
    a = inputs.tensor(M, K, 31, 0)
    b = inputs.tensor(K, N, 31, 1)
    from fp16_gemm_relu_gb300 import gemm_relu_host

    c = gemm_relu_host(a, b)
    assert_parity(c.view(np.uint16), oracle_ref(a, b, True), K, True, where="host entry")
    # odd host leading dimension on the output
    out = np.zeros((M, N + 3), np.float16)[:, :N]
    gemm_relu_host(a, b, out=out)
    np.testing.assert_array_equal(out.view(np.uint16), c.view(np.uint16))


@pytest.mark.parametrize("M,N,K", [(2500, 300, 200), (4100, 264, 1000)])
def test_host_entry_point_multi_panel(M, N, K):
    # several row panels (copies of A and C overlap the panel GEMMs), odd host strides,
    # a ragged last panel
    from fp16_gemm_relu_gb300 import gemm_relu_host

    a = inputs.tensor(M, K, 33, 0)
    b = inputs.tensor(K, N, 33, 1)
    a_host = inputs.embed(a, K + 3)[:, :K]
    out = np.full((M, N + 5), np.nan, np.float16)
    gemm_relu_host(a_host, b, out=out[:, :N])
    assert np.isnan(out[:, N:]).all()
    assert_parity(np.ascontiguousarray(out[:, :N]).view(np.uint16), oracle_ref(a, b, True), K,
                  True, where="host multi-panel")


def test_torch_wrapper_and_views():
    from fp16_gemm_relu_gb300 import gemm_relu

    M, N, K = 200, 300, 400
    a = inputs.tensor(M, K, 37, 0)
    b = inputs.tensor(K, N, 37, 1)
    A = _dev(inputs.embed(a, K + 8))[:, :K]
    B = _dev(b)
    C = gemm_relu(A, B)
    torch.cuda.synchronize()
    assert_parity(C.cpu().numpy().view(np.uint16), oracle_ref(a, b, True), K, True)
    with pytest.raises(TypeError):
        gemm_relu(A.float(), B)


@pytest.mark.parametrize("M,N,K,lda,opts", [
    (4095, 200, 1000, 1001, {"pair": 1, "a_in_place": 1}),
    (4096, 300, 777, 779, {"pair": 1, "split_k": 3, "a_in_place": 1}),
    (4095, 136, 64, 65, {"pair": 1, "a_in_place": 1}),  # K in one k-block, padding after rows
    (8190, 100, 300, 313, {"pair": 1, "split_k": 1, "a_in_place": 1}),
    (4000, 257, 2000, 2003, {"pair": 1, "max_ctas": 6, "a_in_place": 1}),  # several tiles/cluster
])
def test_a_read_by_row_classes(M, N, K, lda, opts):
    # On request, A with a leading dimension that is not a multiple of 8 is read in place
    # through 16 row classes (no repack): each class's K windows start up to 15 elements early, the first
    # window comes from a zero-padded copy, and the partial sums pass through the workspace
    # in class-major row order.  A's padding holds NaN, so a read outside A's rows would show.
    st, plan = binding.tg_plan_query(0x100000, 0x200000, 0x300000, M, N, K, lda, N, N, 152, opts)
    assert st == binding.TG_OK and plan["a_row_classes"] == 16 and plan["repack_a"] == 0
    a = inputs.tensor(M, K, 71, 0)
    b = inputs.tensor(K, N, 71, 1)
    c, pad_ok = run_gpu(a, b, True, opts, lda=lda)
    assert pad_ok
    assert_parity(c, oracle_ref(a, b, True), K, True, where=f"row classes {M}x{N}x{K} lda={lda}")
    ai = inputs.tensor(M, K, 72, 0, "int")
    bi = inputs.tensor(K, N, 72, 1, "int")
    ci, _ = run_gpu(ai, bi, True, opts, lda=lda, ldb=N + 3, ldc=N + 1)
    np.testing.assert_array_equal(ci, oracle.gemm_relu(ai, bi, relu=True, want=("f32",))["out16_f32acc"])


@pytest.mark.parametrize("M,N,K,lda,ldb,split", [
    (1000, 700, 3000, 3001, 703, 3),
    (4095, 300, 8000, 8003, 301, 4),
    (300, 1030, 5000, 5005, 1033, 2),
])
def test_repack_overlap_matches_sequential(M, N, K, lda, ldb, split):
    # With unaligned operands and split-K, each split's slice of A and B is copied on a
    # library stream while the GEMMs of earlier splits run.  The GEMM of each split and the
    # ordered reduction are the same as with the copies first, so the outputs must agree bit
    # for bit, and with the oracle; calls in a row reuse the streams and the scratch pool.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    opts = {"split_k": split}
    st, plan = binding.tg_plan_query(0x100000, 0x200000, 0x300000, M, N, K, lda, ldb, N, sms, opts)
    assert st == binding.TG_OK and plan["repack_overlap"] == 1 and plan["split_k"] == split
    a = inputs.tensor(M, K, 81, 0)
    b = inputs.tensor(K, N, 81, 1)
    seq, ok1 = run_gpu(a, b, True, {"split_k": split, "repack_overlap": -1}, lda=lda, ldb=ldb)
    outs = [run_gpu(a, b, True, opts, lda=lda, ldb=ldb) for _ in range(3)]
    assert ok1 and all(ok for _, ok in outs)
    for c, _ in outs:
        np.testing.assert_array_equal(c, seq)
    assert_parity(seq, oracle_ref(a, b, True), K, True, where=f"overlap {M}x{N}x{K}")
    ai = inputs.tensor(M, K, 82, 0, "int")
    bi = inputs.tensor(K, N, 82, 1, "int")
    ci, _ = run_gpu(ai, bi, True, opts, lda=lda, ldb=ldb, ldc=N + 5)
    np.testing.assert_array_equal(ci, oracle.gemm_relu(ai, bi, relu=True, want=("f32",))["out16_f32acc"])


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,expect", [
    # short K: the default keeps single-CTA 128 x 256 tiles
    (4096, 4096, 512, 512, 4096, 4096, {"cta_pair": 0, "split_k": 1}),
    # long K, aligned C, a last wave of at most half the clusters: one K pass, tail split
    (2048, 3072, 16384, 16384, 3072, 3072, {"cta_pair": 1, "split_k": 1, "tail": True}),
    # unaligned strides on small problems: a few overlapped splits, not 13 to 32
    (1000, 100, 8192, 8195, 103, 101, {"repack_b": 1, "max_split": 4}),
    (1, 4096, 8192, 8195, 4099, 4097, {"repack_b": 1, "max_split": 4}),
])
def test_cost_model_defaults_parity(M, N, K, lda, ldb, ldc, expect):
    # the plans the cost model picks for these shape classes (pinned on the host side too),
    # run by default and compared with the oracle over every output; integer inputs bit for bit
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = binding.tg_plan_query(0x100000, 0x200000, 0x300000, M, N, K, lda, ldb, ldc, sms)
    assert st == binding.TG_OK
    for k in ("cta_pair", "split_k", "repack_b"):
        if k in expect:
            assert plan[k] == expect[k], (k, plan)
    if expect.get("tail"):
        assert plan["tail_tiles"] > 0, plan
    if "max_split" in expect:
        assert 1 <= plan["split_k"] <= expect["max_split"], plan
    a = inputs.tensor(M, K, 97, 0)
    b = inputs.tensor(K, N, 97, 1)
    c, pad_ok = run_gpu(a, b, True, None, lda=lda, ldb=ldb, ldc=ldc)
    assert pad_ok
    assert_parity(c, oracle_ref(a, b, True), K, True, where=f"default plan {M}x{N}x{K}")
    ai = inputs.tensor(M, K, 98, 0, "int")
    bi = inputs.tensor(K, N, 98, 1, "int")
    ci, _ = run_gpu(ai, bi, True, None, lda=lda, ldb=ldb, ldc=ldc)
    np.testing.assert_array_equal(ci, oracle.gemm_relu(ai, bi, relu=True, want=("f32",))["out16_f32acc"])


def test_large_unaligned_operands_copied_first():
    # one K pass with both operands copied first: the copy takes four 32-chunk items per warp
    # pass (all loads before the stores).  Odd leading dimensions and a 2-byte-aligned A.
    M = N = K = 4096
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = binding.tg_plan_query(0x100002, 0x200000, 0x300000, M, N, K, K + 3, N + 3, N + 1,
                                     sms)
    assert st == binding.TG_OK and plan["repack_a"] == 1 and plan["repack_b"] == 1
    assert plan["split_k"] == 1 and plan["repack_overlap"] == 0, plan
    a = inputs.tensor(M, K, 99, 0)
    b = inputs.tensor(K, N, 99, 1)
    c, pad_ok = run_gpu(a, b, True, None, lda=K + 3, ldb=N + 3, ldc=N + 1, a_off=1)
    assert pad_ok
    rows = np.array([0, 1, 7, 8, 2047, 4094, 4095])
    assert_parity(c[rows], oracle.gemm_relu(a, b, relu=True, rows=rows), K, True,
                  where="copies first, 4096^3")
    ai = inputs.tensor(M, K, 100, 0, "int")
    bi = inputs.tensor(K, N, 100, 1, "int")
    ci, _ = run_gpu(ai, bi, True, None, lda=K + 3, ldb=N + 3, ldc=N + 1, a_off=1)
    np.testing.assert_array_equal(
        ci[rows], oracle.gemm_relu(ai, bi, relu=True, rows=rows, want=("f32",))["out16_f32acc"])
