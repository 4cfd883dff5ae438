"""Backward of relu(A·B) on the GPU: transposed-operand GEMMs (every trans_a / trans_b
combination, both kernels, split-K, repacked operands), the relu-backward kernel, and the
torch.autograd.Function built on them, all against the oracle."""

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


def gemm_t(a_stored, b_stored, ta, tb, M, N, K, options=None, pad=0, act=0):
    lda = a_stored.shape[1] + pad
    ldb = b_stored.shape[1] + pad
    A = torch.from_numpy(inputs.embed(a_stored, lda, fill=np.nan)).cuda()
    B = torch.from_numpy(inputs.embed(b_stored, ldb, fill=np.nan)).cuda()
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    st = binding.tg_gemm_f16_t(ta, tb, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda,
                               ldb, N, act, 0, 0, 0, options,
                               torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    return C.cpu().numpy().view(np.uint16)


OPTS = [None, {"pair": 1}, {"pair": -1, "block_n": 192}, {"pair": -1, "split_k": 3},
        {"pair": 1, "split_k": 2, "max_ctas": 4}]


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("tb", [0, 1])
@pytest.mark.parametrize("opts", OPTS, ids=lambda o: "default" if o is None else
                         "-".join(f"{k}{v}" for k, v in o.items()))
def test_transposed_operands(ta, tb, opts):
    M, N, K = 333, 527, 1030
    a = inputs.tensor(M, K, 90, 0)
    b = inputs.tensor(K, N, 90, 1)
    a_st = np.ascontiguousarray(a.T) if ta else a
    b_st = np.ascontiguousarray(b.T) if tb else b
    got = gemm_t(a_st, b_st, ta, tb, M, N, K, opts, pad=8)
    assert_parity(got, oracle.gemm_relu(a, b, relu=False), K, relu=False,
                  where=f"ta={ta} tb={tb} {opts}")


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
def test_transposed_integer_bitwise_and_unaligned(ta, tb):
    M, N, K = 200, 300, 700
    a = inputs.tensor(M, K, 91, 0, "int")
    b = inputs.tensor(K, N, 91, 1, "int")
    a_st = np.ascontiguousarray(a.T) if ta else a
    b_st = np.ascontiguousarray(b.T) if tb else b
    want = oracle.gemm_relu(a, b, relu=True)["out16_f32acc"]
    for pad in (0, 3):  # pad=3: odd leading dimensions, operands are repacked
        got = gemm_t(a_st, b_st, ta, tb, M, N, K, pad=pad, act=1)
        np.testing.assert_array_equal(got, want)


def test_relu_backward_kernel_bitwise():
    M, N = 257, 301
    C = inputs.tensor(M, N, 92, 0)
    C[0, :8] = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 2 ** -24, -1, 1], np.float16)
    dC = inputs.tensor(M, N, 93, 1)
    dC_t = torch.from_numpy(dC).cuda()
    C_t = torch.from_numpy(C).cuda()
    dZ = torch.full((M, N + 5), float("nan"), dtype=torch.float16, device="cuda")
    st = binding.tg_relu_backward_f16(dC_t.data_ptr(), C_t.data_ptr(), dZ.data_ptr(), M, N, N,
                                      N, N + 5, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK
    torch.cuda.synchronize()
    out = dZ.cpu().numpy()
    np.testing.assert_array_equal(out[:, :N].view(np.uint16), oracle.relu_backward(dC, C))
    assert np.isnan(out[:, N:]).all()


@pytest.mark.parametrize("M,N,ld", [(257, 259, 264), (256, 1024, 1024), (9, 5, 8), (1, 8, 8)])
def test_relu_backward_vector_path_every_pattern(M, N, ld):
    # 16-byte-aligned rows take the vectorised kernel (eight rows per thread, a tail thread for
    # the last N mod 8 columns).  C holds every fp16 bit pattern in turn (NaNs, infinities,
    # signed zeros, subnormals), so the mask is pinned bit for bit on that path too; the padding
    # of dZ stays untouched.
    pats = np.arange(M * N, dtype=np.int64) % 65536
    C = np.zeros((M, ld), np.uint16)
    C[:, :N] = pats.reshape(M, N).astype(np.uint16)
    dC = np.zeros((M, ld), np.float16)
    dC[:, :N] = inputs.tensor(M, N, 94, 0)
    C_t = torch.from_numpy(C.view(np.float16)).cuda()
    dC_t = torch.from_numpy(dC).cuda()
    dZ = torch.full((M, ld + 8), float("nan"), dtype=torch.float16, device="cuda")
    st = binding.tg_relu_backward_f16(dC_t.data_ptr(), C_t.data_ptr(), dZ.data_ptr(), M, N, ld,
                                      ld, ld + 8, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK
    torch.cuda.synchronize()
    out = dZ.cpu().numpy()
    want = oracle.relu_backward(np.ascontiguousarray(dC[:, :N]),
                                np.ascontiguousarray(C[:, :N].view(np.float16)))
    np.testing.assert_array_equal(out[:, :N].view(np.uint16), want)
    assert np.isnan(out[:, N:]).all()


@pytest.mark.parametrize("M,N,K", [(300, 520, 777), (1024, 768, 2048)])
def test_autograd_function(M, N, K):
    from fp16_gemm_relu_gb300.autograd import relu_matmul

    a = inputs.tensor(M, K, 94, 0)
    b = inputs.tensor(K, N, 94, 1)
    dc = inputs.tensor(M, N, 95, 1)
    A = torch.from_numpy(a).cuda().requires_grad_(True)
    B = torch.from_numpy(b).cuda().requires_grad_(True)
    C = relu_matmul(A, B)
    C.backward(torch.from_numpy(dc).cuda())
    torch.cuda.synchronize()
    c = C.detach().cpu().numpy()
    assert_parity(c.view(np.uint16), oracle.gemm_relu(a, b), K, True, where="forward")
    ref = oracle.relu_matmul_backward(a, b, c, dc)
    assert_parity(A.grad.cpu().numpy().view(np.uint16), ref["dA"], N, relu=False, where="dA")
    assert_parity(B.grad.cpu().numpy().view(np.uint16), ref["dB"], M, relu=False, where="dB")
