"""Failure detection without a GPU fault: the first producer of the grid drops one pipeline
stage (no load, no arrival), so the MMA thread's bounded wait on it runs out.  The kernel must
record the timeout in the device error word, drain what is in flight, free tensor memory and
return; the host reads TG_ERR_TIMEOUT; the next call on the same context is correct."""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs

from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("pair", [-1, 1], ids=["single_cta", "cta_pair"])
def test_dropped_stage_times_out_and_context_survives(pair):
    from fp16_gemm_relu_gb300 import build

    build.build()
    torch.cuda.set_device(0)
    binding.tg_device_error_check(clear=True)
    M, N, K = 256, 512, 2048
    a = inputs.tensor(M, K, 3, 0)
    b = inputs.tensor(K, N, 3, 1)
    A = torch.from_numpy(a).cuda()
    B = torch.from_numpy(b).cuda()
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    opts = {"debug_flags": binding.TG_DEBUG_DROP_FIRST_STAGE, "timeout_ms": 200, "pair": pair}
    st = binding.tg_gemm_relu_f16_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                                     1, opts, s)
    assert st == binding.TG_OK  # queued; the failure is only visible after it ran
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_ERR_TIMEOUT
    assert word & 1 and ((word >> 8) & 0xFF) in (1, 2, 3)
    # the context is still usable and the error word was cleared
    st, word = binding.tg_device_error_check(clear=False)
    assert st == binding.TG_OK and word == 0
    st = binding.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N, 1, s)
    assert st == binding.TG_OK
    torch.cuda.synchronize()
    ref = oracle.gemm_relu(a, b, relu=True)
    assert_parity(C.cpu().numpy().view(np.uint16), ref, K, True, where="after timeout")
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK and word == 0


def test_host_entry_reports_clean_status():
    M, N, K = 64, 64, 64
    a = inputs.tensor(M, K, 4, 0)
    b = inputs.tensor(K, N, 4, 1)
    out = np.empty((M, N), np.float16)
    st = binding.tg_gemm_relu_f16_host(a.ctypes.data, b.ctypes.data, out.ctypes.data, M, N, K,
                                       K, N, N, 1, 0)
    assert st == binding.TG_OK


@pytest.mark.parametrize("fmt", ["int4", "nf4"])
@pytest.mark.parametrize("kernel", ["swapped", "swapped_tmem", "single_cta", "cta_pair",
                                    "decode_first"])
def test_dequant_kernels_dropped_stage_times_out(fmt, kernel):
    # the same injected fault in the three dequantising GEMM kernels: their waits are bounded
    # like the fp16 kernels'; after the timeout the next call on the context is correct
    from fp16_gemm_relu_gb300 import build

    from tests.test_gpu_w4 import check, make, run_w4

    build.build()
    torch.cuda.set_device(0)
    binding.tg_device_error_check(clear=True)
    # "swapped_tmem": 64 rows of A, weights decoded into tensor memory on request
    M, N, K, G = (64 if kernel == "swapped_tmem" else 256), 512, 2048, 128
    a, Wq, S = make(M, N, K, G, 41)
    # "decode_first": the fp16 GEMM after the decode pass takes the injected fault
    base = {"swapped": {"swap_ab": 1}, "swapped_tmem": {"swap_ab": 1, "tmem_decode": 1},
            "decode_first": {"dequant_first": 1},
            "single_cta": {"swap_ab": -1, "block_n": 128},
            "cta_pair": {"swap_ab": -1, "pair": 1}}[kernel]
    opts = dict(base, debug_flags=binding.TG_DEBUG_DROP_FIRST_STAGE, timeout_ms=200)
    fn = binding.tg_gemm_w4a16_f16 if fmt == "int4" else binding.tg_gemm_nf4a16_f16
    A = torch.from_numpy(a).cuda()
    Q = torch.from_numpy(Wq.view(np.int32)).cuda()
    Sc = torch.from_numpy(S).cuda()
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    st = fn(A.data_ptr(), Q.data_ptr(), Sc.data_ptr(), C.data_ptr(), M, N, K, K, Wq.shape[1],
            S.shape[1], N, G, 1, 0, 0, 0, opts, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK  # queued; the failure is only visible after it ran
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_ERR_TIMEOUT, (st, hex(word))
    assert word & 1 and ((word >> 8) & 0xFF) in (1, 2, 3)
    st, word = binding.tg_device_error_check(clear=False)
    assert st == binding.TG_OK and word == 0
    got = run_w4(a, Wq, S, N, G, act=1, options=base, fmt=fmt)
    check(got, a, Wq, S, N, G, "relu", fmt=fmt)
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK and word == 0
