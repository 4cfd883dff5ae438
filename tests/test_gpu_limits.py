"""Size limits: an output with more than 2^32 elements (64-bit offsets in the TMA-stored body,
in the plain-store column tail and in C's padding), and a very long K (deep split-K
accumulation), each compared with the oracle on sampled rows and columns."""

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


def _check(got_bits, a, b, rows, cols, relu=True):
    ref = oracle.gemm_relu(a, b, relu=relu, rows=rows, cols=cols)
    c = compare(got_bits, ref, a.shape[1], relu=relu)
    assert c["out_of_tol"] == 0 and (not relu or c["zero_rule"] == 0), c


def test_output_beyond_2_pow_32_elements():
    M, N, K = 65536, 65541, 64           # N % 8 == 5: five columns go through the tail stores
    ldc = 65544
    assert M * ldc > 2 ** 32
    a = inputs.tensor(M, K, 101, 0)
    b = inputs.tensor(K, N, 101, 1)
    A = torch.from_numpy(a).cuda()
    B = torch.zeros((K, ldc), dtype=torch.float16, device="cuda")
    B[:, :N] = torch.from_numpy(b).cuda()
    canary = 0x7E5A
    C = torch.full((M, ldc), canary, dtype=torch.int16, device="cuda")
    st = binding.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, ldc, ldc,
                                  binding.TG_EPILOGUE_RELU, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 32767, 32768, M - 2, M - 1], rng.integers(0, M, 40)]))
    cols = np.unique(np.concatenate([[0, 7, 8, 65535], np.arange(65528, N),
                                     rng.integers(0, N, 40)]))
    sub = C[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()]
    got = sub.cpu().numpy().view(np.uint16)
    _check(got, a, b, rows, cols)
    pad = C[torch.from_numpy(rows).cuda()][:, N:].cpu().numpy().view(np.uint16)
    assert (pad == canary).all()  # the padding past column N is never written


def test_very_long_k():
    M, N, K = 96, 136, 1_000_003
    a = inputs.tensor(M, K, 102, 0)
    b = inputs.tensor(K, N, 102, 1)
    lda = -(-K // 8) * 8
    A = torch.zeros((M, lda), dtype=torch.float16, device="cuda")
    A[:, :K] = torch.from_numpy(a).cuda()
    B = torch.from_numpy(b).cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    st = binding.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, N, N,
                                  binding.TG_EPILOGUE_RELU, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    rows = np.array([0, 17, 50, 95])
    got = C.cpu().numpy().view(np.uint16)[rows]
    _check(got, a, b, rows, np.arange(N))
