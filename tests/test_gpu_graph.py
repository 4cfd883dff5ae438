"""Capture of the asynchronous entry points in a CUDA graph and replay.  The first call on a
device sets up library state (pool, attributes), so each path runs once eagerly before the
capture; inside the capture, the stream-ordered scratch of the repack + split-K path becomes
graph allocation nodes.  Replays must reproduce the eager results bit for bit."""

import numpy as np
import pytest

from fp16_gemm_relu_gb300 import binding, inputs

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


def _calls(A, B, C3, bias, M, N, K, stream):
    a, b = A.data_ptr(), B.data_ptr()
    sts = [
        binding.tg_gemm_relu_f16(a, b, C3[0].data_ptr(), M, N, K, K, N, N, 1, stream),
        binding.tg_gemm_relu_f16_ex(a, b, C3[1].data_ptr(), M, N, K, K, N, N, 1,
                                    {"split_k": 3, "force_repack": 1}, stream),
        binding.tg_gemm_f16_epilogue(a, b, C3[2].data_ptr(), M, N, K, K, N, N, 3,
                                     bias.data_ptr(), 0, 0, None, stream),
    ]
    for st in sts:
        assert st == binding.TG_OK, binding.tg_status_string(st)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (333, 520, 1030)])
def test_capture_and_replay(M, N, K):
    A = torch.from_numpy(inputs.tensor(M, K, 95, 0)).cuda()
    B = torch.from_numpy(inputs.tensor(K, N, 95, 1)).cuda()
    bias = torch.from_numpy(inputs.tensor(1, N, 96, 0).ravel()).cuda()
    eager = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(3)]
    _calls(A, B, eager, bias, M, N, K, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want = [c.cpu().numpy().view(np.uint16) for c in eager]

    out = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _calls(A, B, out, bias, M, N, K, side.cuda_stream)  # warm-up on the capturing stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=side):
        _calls(A, B, out, bias, M, N, K, side.cuda_stream)
    for rep in range(3):
        for c in out:
            c.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for c, w in zip(out, want):
            np.testing.assert_array_equal(c.cpu().numpy().view(np.uint16), w, err_msg=f"replay {rep}")
