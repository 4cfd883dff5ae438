"""Parity at the five named workloads' full sizes, in the launch configuration bench.py times
(the default plan through tg_gemm_relu_f16, natural leading dimensions).

The two small workloads are compared with the oracle element by element.  The large ones are
compared on a sampled grid of outputs (edge rows/columns plus seeded random ones) that the
oracle computes one by one, and on properties of the whole output: no negative or non-finite
value, bitwise determinism, and exactness on integer-valued inputs of the same shape."""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs, workloads

from tests.parity import assert_parity, compare

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


def run_default(a, b):
    M, K = a.shape
    N = b.shape[1]
    A = torch.from_numpy(a).cuda()
    B = torch.from_numpy(b).cuda()
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    st = binding.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                                  binding.TG_EPILOGUE_RELU, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK
    torch.cuda.synchronize()
    return C


def sample_grid(M, N, count, seed):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 1, M // 2, M - 2, M - 1],
                                     rng.integers(0, M, count)]).clip(0, M - 1))
    cols = np.unique(np.concatenate([[0, 1, N // 2, N - 2, N - 1],
                                     rng.integers(0, N, count)]).clip(0, N - 1))
    return rows, cols


@pytest.mark.parametrize("name", ["square256", "square2048"])
def test_small_workloads_full_parity(name):
    wl = workloads.get(name)
    a, b = wl.make_a(), wl.make_b()
    got = run_default(a, b).cpu().numpy().view(np.uint16)
    ref = oracle.gemm_relu(a, b, relu=True)
    c = assert_parity(got, ref, wl.K, True, where=name)
    assert c["rel_fro"] < 1e-3, c  # fp16 output rounding alone is ~2e-4


@pytest.mark.parametrize("name", ["square8192", "skinny64x28672x8192", "ragged4095x3073x65537"])
def test_large_workloads_sampled_parity(name):
    wl = workloads.get(name)
    a, b = wl.make_a(), wl.make_b()
    C = run_default(a, b)
    C2 = run_default(a, b)
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16)), "not deterministic"
    full = C.cpu().numpy().view(np.uint16)
    assert not (full & 0x8000).any(), "negative or -0 output under relu"
    assert not ((full & 0x7C00) == 0x7C00).any(), "non-finite output"
    rows, cols = sample_grid(wl.M, wl.N, 60, wl.seed)
    ref = oracle.gemm_relu(a, b, relu=True, rows=rows, cols=cols)
    got = full[np.ix_(rows, cols)]
    c = assert_parity(got, ref, wl.K, True, where=name)
    assert c["rel_fro"] < 1e-3, c  # fp16 output rounding alone is ~2e-4


@pytest.mark.parametrize("name", ["square8192", "ragged4095x3073x65537"])
def test_large_workloads_integer_inputs_bitwise(name):
    wl = workloads.get(name)
    a = inputs.tensor(wl.M, wl.K, wl.seed, 0, "int")
    b = inputs.tensor(wl.K, wl.N, wl.seed, 1, "int")
    full = run_default(a, b).cpu().numpy().view(np.uint16)
    rows, cols = sample_grid(wl.M, wl.N, 40, wl.seed + 100)
    ref = oracle.gemm_relu(a, b, relu=True, rows=rows, cols=cols, want=("f32",))
    np.testing.assert_array_equal(full[np.ix_(rows, cols)], ref["out16_f32acc"])


def test_default_tail_split_with_ragged_edges():
    # 20 x 16 = 320 pair tiles: four full waves of 76 clusters, then 16 tiles that the default
    # plan runs as 32 K halves.  M, N and K all end in partial tiles (5000 = 19*256 + 136,
    # 4000 = 15*256 + 160, 1000 = 15*64 + 40), so the split tiles include edge tiles and the
    # second K half ends in a partial k-block.
    M, N, K = 5000, 4000, 1000
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = binding.tg_plan_query(0x1000, 0x2000, 0x3000, M, N, K, K, N, N, sms)
    assert st == binding.TG_OK and plan["cta_pair"] == 1
    clusters = plan["grid"] // 2
    r = (plan["tiles_m"] * plan["tiles_n"]) % clusters
    assert plan["tail_tiles"] == (r if 0 < 2 * r <= clusters else 0)
    a = inputs.tensor(M, K, 61, 0)
    b = inputs.tensor(K, N, 61, 1)
    C = run_default(a, b)
    assert torch.equal(C.view(torch.int16), run_default(a, b).view(torch.int16)), "not deterministic"
    full = C.cpu().numpy().view(np.uint16)
    # rows and columns of the last tile row/column (where the split tiles sit) plus a sample
    rows = np.unique(np.concatenate([np.arange(4864, M, 7), sample_grid(M, N, 30, 62)[0]]))
    cols = np.unique(np.concatenate([np.arange(3840, N, 5), sample_grid(M, N, 30, 63)[1]]))
    ref = oracle.gemm_relu(a, b, relu=True, rows=rows, cols=cols)
    assert_parity(full[np.ix_(rows, cols)], ref, K, True, where="tail split, ragged")
    ai = inputs.tensor(M, K, 64, 0, "int")
    bi = inputs.tensor(K, N, 64, 1, "int")
    fi = run_default(ai, bi).cpu().numpy().view(np.uint16)
    refi = oracle.gemm_relu(ai, bi, relu=True, rows=rows, cols=cols, want=("f32",))
    np.testing.assert_array_equal(fi[np.ix_(rows, cols)], refi["out16_f32acc"])
