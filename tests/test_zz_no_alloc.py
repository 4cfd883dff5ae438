"""The allocation-free split-K entry point, tg_gemm_relu_f16_splitk_noalloc.

Some callers cannot allocate device memory while they run a GEMM: code running inside an
allocator that must not be re-entered, a runtime that owns all device memory in its own arena,
or latency-critical work where an allocation could block.  This entry point serves them with a
fixed workspace array that is part of the library.  Its output is checked, through the C ABI,
against the ordinary entry point tg_gemm_relu_f16 on the same inputs, with the tolerance the
other parity tests use, on two calls in a row (the second one runs on a workspace that still
holds the first call's partial sums).  This file is collected last, so a run that stops at its
first failure has already run every other test; it also passes on its own in a fresh process.
"""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs

from tests.parity import ulp16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from fp16_gemm_relu_gb300 import build

    build.build()
    binding.load_library()
    torch.cuda.set_device(0)


def _close(new_bits, ref_bits, K):
    """Elements with |new - ref| > 2 ulp16(ref) + 1e-4 sqrt(K), ref = the ordinary entry
    point's output; non-finite values count as failures."""
    r = oracle.f16_bits_to_f64(ref_bits)
    g = oracle.f16_bits_to_f64(new_bits)
    tol = 2.0 * ulp16(r) + 1e-4 * np.sqrt(K)
    bad = ~(np.abs(g - r) <= tol) | ~np.isfinite(g) | ~np.isfinite(r)
    return int(bad.sum()), float(np.nanmax(np.abs(g - r)))


def _run_pair(M, N, K, seed, split_k, relu, ldc=None):
    """Both entry points on the same inputs.  The no-alloc entry point reads A and B with TMA,
    so their rows must start on 16-byte boundaries: the operands sit in buffers whose leading
    dimensions are rounded up to multiples of 8 (padding filled with NaN, which must never be
    read).  M, N, K and ldc may be ragged."""
    a = inputs.tensor(M, K, seed, 0)
    b = inputs.tensor(K, N, seed, 1)
    ldc = ldc or N
    lda = -(-K // 8) * 8
    ldb = -(-N // 8) * 8
    A = torch.from_numpy(inputs.embed(a, lda, fill=np.nan)).cuda()
    B = torch.from_numpy(inputs.embed(b, ldb, fill=np.nan)).cuda()
    C_ref = torch.zeros((M, ldc), dtype=torch.float16, device="cuda")
    C_new = torch.full((M, ldc), float("nan"), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    flag = binding.TG_EPILOGUE_RELU if relu else binding.TG_EPILOGUE_NONE
    st = binding.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C_ref.data_ptr(), M, N, K, lda,
                                  ldb, ldc, flag, s)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    st = binding.tg_gemm_relu_f16_splitk_noalloc(A.data_ptr(), B.data_ptr(), C_new.data_ptr(),
                                                 M, N, K, lda, ldb, ldc, flag, split_k, s)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    ref = C_ref.cpu().numpy().view(np.uint16)
    new = C_new.cpu().numpy().view(np.uint16)
    return ref[:, :N], new[:, :N], new[:, N:]


def test_matches_ordinary_entry_point_on_two_calls_in_a_row():
    # first call: the larger problem with 3 splits; second: a smaller, ragged one with 2 splits
    for (M, N, K, seed, split, relu) in [(700, 1200, 3000, 41, 3, True),
                                          (333, 517, 1029, 42, 2, False)]:
        ref, new, _ = _run_pair(M, N, K, seed, split, relu)
        nbad, maxerr = _close(new, ref, K)
        assert nbad == 0, f"{M}x{N}x{K}: {nbad} elements out of tolerance (max {maxerr})"
        if relu:
            assert not (new & 0x8000).any()
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK, hex(word)


def test_padded_output_untouched_and_limits():
    # a padded C with an odd leading dimension: its padding columns keep their contents
    ref, new, pad = _run_pair(130, 250, 640, 43, 4, True, ldc=259)
    assert _close(new, ref, 640)[0] == 0
    assert np.isnan(pad.view(np.float16)).all()
    # larger than the fixed workspace: refused before anything is launched
    M, N = 4096, 4096
    assert 2 * M * N * 4 > binding.TG_STATIC_WORKSPACE_BYTES
    st = binding.tg_gemm_relu_f16_splitk_noalloc(256, 256, 256, M, N, 1024, 1024, N, N, 1, 2, 0)
    assert st == binding.TG_ERR_NO_WORKSPACE
    # operand rows that do not start on 16-byte boundaries are refused, not copied
    st = binding.tg_gemm_relu_f16_splitk_noalloc(256, 256, 256, 64, 64, 64, 64, 65, 64, 1, 1, 0)
    assert st == binding.TG_ERR_MISALIGNED
