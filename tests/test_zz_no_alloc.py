"""The allocation-free split-K entry point, tg_gemm_relu_f16_splitk_noalloc.

Some callers cannot allocate device memory while they run a GEMM: code running inside an
allocator that must not be re-entered, a runtime that owns all device memory in its own arena,
or latency-critical work where an allocation could block.  This entry point serves them with a
fixed workspace array that is part of the library.

Its output is checked through the C ABI on two calls in a row (the second one runs on a
workspace that still holds the first call's partial sums):
  - against the oracle, element by element, with the tolerance and zero rule of every other
    parity test (tests/parity.py), so that a fault shared by the split-K kernels cannot hide;
  - against the ordinary entry point tg_gemm_relu_f16 on the same inputs, within the same
    tolerance.
The planning branches where this entry point differs from the ordinary one are covered too:
K == 0 (a memset of +0 that leaves C's padding alone), split_k == 0 (two splits) and a split
count larger than the number of 64-wide K blocks (clamped so that every split is non-empty).

This file is collected last, so a run that stops at its first failure has already run every
other test; it also passes on its own in a fresh process.
"""

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs

from tests.parity import assert_parity, ulp16

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


def _close(new_bits, ref_bits, K):
    """Elements with |new - ref| > 2 ulp16(ref) + 1e-4 sqrt(K), ref = the ordinary entry
    point's output; non-finite values count as failures."""
    r = oracle.f16_bits_to_f64(ref_bits)
    g = oracle.f16_bits_to_f64(new_bits)
    tol = 2.0 * ulp16(r) + 1e-4 * np.sqrt(max(K, 1))
    bad = ~(np.abs(g - r) <= tol) | ~np.isfinite(g) | ~np.isfinite(r)
    return int(bad.sum()), float(np.nanmax(np.abs(g - r))) if g.size else 0.0


def _run_pair(M, N, K, seed, split_k, relu, ldc=None):
    """Both entry points on the same inputs; returns (a, b, ordinary C, no-alloc C, no-alloc
    C's padding columns).  The no-alloc entry point reads A and B with TMA, so their rows must
    start on 16-byte boundaries: the operands sit in buffers whose leading dimensions are
    rounded up to multiples of 8 (padding filled with NaN, which must never be read).  M, N,
    K and ldc may be ragged."""
    a = inputs.tensor(M, K, seed, 0)
    b = inputs.tensor(K, N, seed, 1)
    ldc = ldc or N
    lda = max(-(-K // 8) * 8, 8)
    ldb = -(-N // 8) * 8
    A = torch.from_numpy(inputs.embed(a, lda, fill=np.nan)).cuda() if K else \
        torch.full((M, lda), float("nan"), dtype=torch.float16, device="cuda")
    B = torch.from_numpy(inputs.embed(b, ldb, fill=np.nan)).cuda() if K else \
        torch.full((1, ldb), float("nan"), dtype=torch.float16, device="cuda")
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
    return a, b, ref[:, :N], new[:, :N], new[:, N:]


def _check(M, N, K, seed, split_k, relu, ldc=None):
    a, b, ref, new, pad = _run_pair(M, N, K, seed, split_k, relu, ldc)
    where = f"{M}x{N}x{K} split_k={split_k} relu={relu}"
    # against the oracle: the tolerance and zero rule of every parity test
    want = oracle.gemm_relu(a, b, relu=relu)
    assert_parity(new, want, K, relu, where="no-alloc vs oracle " + where)
    # against the ordinary entry point, within the same tolerance
    nbad, maxerr = _close(new, ref, K)
    assert nbad == 0, f"{where}: {nbad} elements out of tolerance vs tg_gemm_relu_f16 ({maxerr})"
    return new, pad


def test_matches_oracle_and_ordinary_entry_point_on_two_calls_in_a_row():
    # first call: the larger problem with 3 splits; second: a smaller, ragged one with 2 splits
    # on a workspace that still holds the first call's partial sums
    _check(700, 1200, 3000, 41, 3, True)
    _check(333, 517, 1029, 42, 2, False)
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK, hex(word)


def test_padded_output_untouched_and_limits():
    # a padded C with an odd leading dimension: its padding columns keep their contents
    _, pad = _check(130, 250, 640, 43, 4, True, ldc=259)
    assert np.isnan(pad.view(np.float16)).all()
    # larger than the fixed workspace: refused before anything is launched
    M, N = 4096, 4096
    assert 2 * M * N * 4 > binding.TG_STATIC_WORKSPACE_BYTES
    st = binding.tg_gemm_relu_f16_splitk_noalloc(256, 256, 256, M, N, 1024, 1024, N, N, 1, 2, 0)
    assert st == binding.TG_ERR_NO_WORKSPACE
    # operand rows that do not start on 16-byte boundaries are refused, not copied
    st = binding.tg_gemm_relu_f16_splitk_noalloc(256, 256, 256, 64, 64, 64, 64, 65, 64, 1, 1, 0)
    assert st == binding.TG_ERR_MISALIGNED


def test_planning_branches():
    # K == 0: C = +0 exactly (the empty sum), padding of a wider ldc untouched
    new, pad = _check(77, 90, 0, 44, 3, True, ldc=97)
    assert (new == 0).all()
    assert np.isnan(pad.view(np.float16)).all()
    # split_k == 0 picks two splits
    _check(200, 300, 1000, 45, 0, True)
    # split_k = 8 with K = 100 (two K blocks): clamped so that each split is non-empty
    _check(150, 260, 100, 46, 8, True)
    # the effective split count below the request (10 K blocks, 6 asked, 5 used)
    _check(129, 131, 640, 47, 6, False)
