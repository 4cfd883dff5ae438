"""Concurrent calls from several host threads (the header promises that every entry point may be
called from several threads at once).  Each thread uses its own stream and output buffers and
repeats calls that exercise the direct path, the operand repack + split-K workspace path (the
library's scratch pool) and the fused epilogue; two threads also use the host-buffer entry
point, whose copy pipeline is shared.  A plan fixes the summation order, so every result must
equal the single-threaded reference bit for bit.  ctypes releases the GIL around foreign calls,
so the library really is entered concurrently."""

import threading

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


def _case(kind, A, B, C, M, N, K, lda, ldb, ldc, bias, stream):
    if kind == "direct":
        return binding.tg_gemm_relu_f16(A, B, C, M, N, K, lda, ldb, ldc, 1, stream)
    if kind == "repack_splitk":
        return binding.tg_gemm_relu_f16_ex(A, B, C, M, N, K, lda, ldb, ldc, 1,
                                           {"split_k": 3, "force_repack": 1}, stream)
    if kind == "epilogue":
        return binding.tg_gemm_f16_epilogue(A, B, C, M, N, K, lda, ldb, ldc, 2, bias, 0, 0, None,
                                            stream)
    raise ValueError(kind)


def test_concurrent_device_calls_match_single_threaded():
    M, N, K = 520, 776, 1000
    a = inputs.tensor(M, K, 91, 0)
    b = inputs.tensor(K, N, 91, 1)
    A = torch.from_numpy(a).cuda()
    B = torch.from_numpy(b).cuda()
    bias = torch.from_numpy(inputs.tensor(1, N, 92, 0).ravel()).cuda()
    kinds = ["direct", "repack_splitk", "epilogue"]
    refs = {}
    for kind in kinds:
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        st = _case(kind, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                   bias.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == binding.TG_OK, binding.tg_status_string(st)
        torch.cuda.synchronize()
        refs[kind] = C.cpu().numpy().view(np.uint16)

    threads, iters = 4, 6
    outs = [[torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
             for _ in range(iters * len(kinds))] for _ in range(threads)]
    streams = [torch.cuda.Stream() for _ in range(threads)]
    errors = []
    start = threading.Barrier(threads)

    def worker(t):
        try:
            start.wait()
            s = streams[t].cuda_stream
            for i in range(iters):
                for j, kind in enumerate(kinds):
                    C = outs[t][i * len(kinds) + j]
                    st = _case(kind, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N,
                               bias.data_ptr(), s)
                    if st != binding.TG_OK:
                        errors.append((t, kind, i, binding.tg_status_string(st),
                                       binding.tg_last_cuda_error()))
        except Exception as e:  # reported below, on the main thread
            errors.append((t, repr(e)))

    ts = [threading.Thread(target=worker, args=(t,)) for t in range(threads)]
    for th in ts:
        th.start()
    for th in ts:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for t in range(threads):
        for i in range(iters):
            for j, kind in enumerate(kinds):
                got = outs[t][i * len(kinds) + j].cpu().numpy().view(np.uint16)
                np.testing.assert_array_equal(got, refs[kind], err_msg=f"thread {t} {kind} #{i}")


def test_concurrent_host_entry_point():
    M, N, K = 1030, 512, 700
    a = inputs.tensor(M, K, 93, 0)
    b = inputs.tensor(K, N, 93, 1)
    ref = np.empty((M, N), np.float16)
    st = binding.tg_gemm_relu_f16_host(a.ctypes.data, b.ctypes.data, ref.ctypes.data, M, N, K,
                                       K, N, N, 1, 0)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    threads = 2
    outs = [[np.full((M, N), np.nan, np.float16) for _ in range(4)] for _ in range(threads)]
    errors = []

    def worker(t):
        s = torch.cuda.Stream()
        for C in outs[t]:
            st = binding.tg_gemm_relu_f16_host(a.ctypes.data, b.ctypes.data, C.ctypes.data, M, N,
                                               K, K, N, N, 1, s.cuda_stream)
            if st != binding.TG_OK:
                errors.append((t, binding.tg_status_string(st)))

    ts = [threading.Thread(target=worker, args=(t,)) for t in range(threads)]
    for th in ts:
        th.start()
    for th in ts:
        th.join()
    assert not errors, errors
    for t in range(threads):
        for C in outs[t]:
            np.testing.assert_array_equal(C.view(np.uint16), ref.view(np.uint16))
