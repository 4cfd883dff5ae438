"""The C-ABI library without a GPU: it loads, exports every declared symbol, and its host-only
logic (argument validation, plan selection, status strings) behaves as documented."""

import ctypes
import os
import re

import pytest

import fp16_gemm_relu_gb300 as tg
from fp16_gemm_relu_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp16_gemm_relu_gb300 import build

    build.build()
    return tg.load_library()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(tg_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "tg_gemm_relu_f16" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for s in range(7):
        assert binding.tg_status_string(s)
    assert binding.tg_status_string(99) == "unknown status"
    assert binding.tg_version() == 300


def test_validation_before_any_device_work(lib):
    # these return from host validation, before any CUDA call
    p = 4096
    assert binding.tg_gemm_relu_f16(p, p, p, -1, 4, 4, 4, 4, 4, 1) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(p, p, p, 4, 4, 4, 3, 4, 4, 1) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(p, p, p, 4, 4, 4, 4, 3, 4, 1) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(p, p, p, 4, 4, 4, 4, 4, 3, 1) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(p, p, p, 4, 4, 4, 4, 4, 4, 2) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(0, p, p, 4, 4, 4, 4, 4, 4, 1) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(p, p, 0, 4, 4, 4, 4, 4, 4, 1) == binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16(p + 1, p, p, 4, 4, 4, 4, 4, 4, 1) == binding.TG_ERR_MISALIGNED
    assert binding.tg_gemm_relu_f16(p, p, p + 1, 4, 4, 4, 4, 4, 4, 1) == binding.TG_ERR_MISALIGNED
    # empty output: a no-op that succeeds
    assert binding.tg_gemm_relu_f16(0, 0, 0, 0, 5, 5, 5, 5, 5, 1) == binding.TG_OK
    assert binding.tg_gemm_relu_f16(0, 0, 0, 5, 0, 5, 5, 1, 1, 1) == binding.TG_OK
    assert binding.tg_gemm_relu_f16_host(0, 0, 0, -3, 1, 1, 1, 1, 1, 1) == binding.TG_ERR_INVALID_ARG
    st, _ = binding.tg_plan_query(p, p, p, 4, 4, 4, 4, 4, 4, 0)
    assert st == binding.TG_ERR_INVALID_ARG
    st, _ = binding.tg_plan_query(p, p, p, 4, 4, 4, 4, 4, 4, 152, {"block_n": 96})
    assert st == binding.TG_ERR_INVALID_ARG


def _plan(M, N, K, **kw):
    opts = kw.pop("options", None)
    return tg.plan(M, N, K, options=opts, **kw)


def test_plan_square_is_one_kernel_pair_tiles(lib):
    p = _plan(8192, 8192, 8192)
    assert p["cta_pair"] == 1
    assert (p["block_m"], p["block_n"], p["block_k"]) == (256, 256, 64)
    assert p["split_k"] == 1 and p["kernels"] == 1
    assert p["tiles_m"] == 32 and p["tiles_n"] == 32 and p["units"] == 1024 + p["tail_tiles"]
    # forward CTA-pair stages hold two 64-k blocks: 3 stages of 64 KB per CTA
    assert p["grid"] == 152 and p["grid"] % 2 == 0 and p["stages"] == 3
    q = _plan(8192, 8192, 8192, options={"pair": -1})
    assert q["cta_pair"] == 0 and (q["block_m"], q["block_n"]) == (128, 256)
    assert q["units"] == 2048 and q["grid"] == 152 and q["stages"] == 4


def test_plan_pair_overrides(lib):
    p = _plan(300, 600, 1500, options={"pair": 1, "max_ctas": 5})
    assert p["cta_pair"] == 1 and p["grid"] == 4 and p["tiles_m"] == 2 and p["tiles_n"] == 3
    st, _ = binding.tg_plan_query(4096, 4096, 4096, 64, 64, 64, 64, 64, 64, 152,
                                  {"pair": 1, "block_n": 128})
    assert st == binding.TG_ERR_INVALID_ARG


def test_plan_short_k_keeps_single_cta_tiles(lib):
    # at K <= 1024 the pair kernel's start and its tail split cost more than they save: on
    # GB300 8192x8192x512 ran 76.8 us on 128x256 tiles against 96.1 us on pair tiles
    for M, N, K in [(8192, 8192, 256), (8192, 8192, 512), (4096, 4096, 1024)]:
        p = _plan(M, N, K)
        assert p["cta_pair"] == 0 and p["split_k"] == 1, (M, N, K, p)


def test_plan_long_k_prefers_the_tail_split_over_split_k(lib):
    # aligned C and a last wave of at most half the clusters: one K pass with the tail split
    # beats two or three K splits through the workspace (2048x8192x65536: 1296 against
    # 1340 us; 12288x512x16384: 150 against 167 us)
    for M, N, K in [(2048, 8192, 65536), (12288, 512, 16384), (2048, 3072, 16384)]:
        p = _plan(M, N, K)
        assert p["cta_pair"] == 1 and p["split_k"] == 1 and p["tail_tiles"] > 0, (M, N, K, p)


def test_plan_unaligned_small_problem_few_splits(lib):
    # an unaligned B on a small problem: every overlapped split is one more GEMM launch and two
    # copies, so the plan keeps the split count low (1000x100x8192: 3 splits ran 57 us, the
    # 13 of a model without that cost 126 us; 1x4096x8192: 81 against 212 us)
    for M, N, K, lda, ldb in [(1000, 100, 8192, 8195, 103), (1, 4096, 8192, 8195, 4099)]:
        p = _plan(M, N, K, lda=lda, ldb=ldb, ldc=N + 1)
        assert p["repack_b"] == 1 and p["split_k"] <= 4, (M, N, K, p)


def test_plan_skinny_fills_the_machine(lib):
    p = _plan(64, 28672, 8192)
    assert p["units"] >= 0.95 * 152 or p["split_k"] > 1
    assert p["grid"] >= 140


def test_plan_ragged_unaligned(lib):
    # odd leading dimensions: A and B are repacked into 128-byte rows, C goes through the fp32
    # workspace
    p = _plan(4095, 3073, 65537)
    assert p["repack_a"] == 1 and p["repack_b"] == 1 and p["workspace_epilogue"] == 1
    assert p["a_row_classes"] == 0 and p["kblocks"] == 1025
    # the copies overlap the GEMMs split by split: per split two copies and one GEMM, then
    # one reduction
    assert p["repack_overlap"] == 1 and p["kernels"] == 3 * p["split_k"] + 1
    q = _plan(4095, 3073, 65537, options={"repack_overlap": -1})
    assert q["repack_overlap"] == 0 and q["kernels"] == 4
    assert p["split_k"] * p["kblocks_per_split"] >= 1025
    assert (p["split_k"] - 1) * p["kblocks_per_split"] < 1025
    ws = 4095 * 65600 * 2 + 65537 * 3136 * 2 + p["split_k"] * 4095 * 3104 * 4
    assert p["workspace_bytes"] >= ws
    # on request, A (32-byte aligned) is read in place through 16 row classes instead
    c = _plan(4095, 3073, 65537, options={"a_in_place": 1})
    assert c["a_row_classes"] == 16 and c["repack_a"] == 0
    assert c["repack_b"] == 1 and c["workspace_epilogue"] == 1 and c["cta_pair"] == 1
    assert c["kernels"] == 4  # first-window copy, B repack, GEMM, reduction
    assert c["tiles_m"] == 16  # 16 classes of 256 rows: no more tiles than 4095 rows need
    assert c["kblocks"] == 1025  # windows start up to 15 elements early: ceil((K + 15) / 64)
    wsc = 16 * 256 * 64 * 2 + 65537 * 3136 * 2 + c["split_k"] * 16 * 256 * 3104 * 4
    assert c["workspace_bytes"] >= wsc and c["workspace_bytes"] < ws
    # not possible: A only 16-byte aligned (a class base would start before A), a forced
    # repack, or an M whose class-major order adds tiles (2000 rows: 16 classes of 125 rows,
    # each in a tile of 256)
    for kw in ({"a_ptr": 256 + 16}, {"options": {"a_in_place": 1, "force_repack": 1}}):
        r = _plan(4095, 3073, 65537, **({"options": {"a_in_place": 1}} | kw))
        assert r["a_row_classes"] == 0 and r["repack_a"] == 1
    g = _plan(2000, 3073, 65537, options={"a_in_place": 1})
    assert g["a_row_classes"] == 0 and g["repack_a"] == 1


def test_plan_alignment_from_pointers(lib):
    a = _plan(256, 256, 256, a_ptr=258)
    assert a["repack_a"] == 1 and a["repack_b"] == 0 and a["workspace_epilogue"] == 0
    c = _plan(256, 256, 256, c_ptr=264)
    assert c["workspace_epilogue"] == 1


def test_plan_overrides(lib):
    p = _plan(1000, 1000, 1000, options={"block_n": 128, "split_k": 3, "max_ctas": 5,
                                          "panel_m": 2, "pair": -1})
    assert p["block_n"] == 128 and p["split_k"] == 3 and p["grid"] == 5 and p["panel_m"] == 2
    assert p["workspace_epilogue"] == 1 and p["units"] == 8 * 8 * 3
    # more splits than K blocks are clamped, and no split is empty
    q = _plan(100, 100, 130, options={"split_k": 50})
    assert q["split_k"] == 3 and q["kblocks_per_split"] == 1
    r = _plan(100, 100, 1000, options={"split_k": 6})
    assert (r["split_k"] - 1) * r["kblocks_per_split"] < r["kblocks"]


def test_plan_k_zero_and_empty(lib):
    assert _plan(10, 10, 0)["kernels"] == 1
    assert _plan(0, 10, 10)["kernels"] == 0


def test_epilogue_argument_errors(lib):
    # rejected by host validation before any device work
    p = 4096
    e = binding.tg_gemm_f16_epilogue
    assert e(p, p, p, 4, 4, 4, 4, 4, 4, 9) == binding.TG_ERR_INVALID_ARG        # activation
    assert e(p, p, p, 4, 4, 4, 4, 4, 4, 1, p + 1) == binding.TG_ERR_MISALIGNED  # bias
    assert e(p, p, p, 4, 4, 4, 4, 4, 4, 1, 0, p, 3) == binding.TG_ERR_INVALID_ARG  # ldr < N
    assert e(p, p, p, 4, 4, 4, 4, 4, 8, 1, 0, p, 4) == binding.TG_ERR_INVALID_ARG  # C alias, ldr != ldc
    assert e(0, 0, 0, 0, 4, 4, 4, 4, 4, 2) == binding.TG_OK                       # empty


def test_w4_argument_errors(lib):
    p = 4096
    def call(*a):
        args = [p, p, p, p, 64, 64, 64, 64, 8, 64, 64, 128]
        for i, v in a:
            args[i] = v
        return binding.tg_gemm_w4a16_f16(*args)
    assert call() == binding.TG_ERR_UNSUPPORTED_DEVICE or call() in (binding.TG_ERR_CUDA, binding.TG_OK)
    assert call((11, 96)) == binding.TG_ERR_INVALID_ARG     # group size not a multiple of 64
    assert call((8, 7)) == binding.TG_ERR_INVALID_ARG       # ldq < ceil(N/8)
    assert call((9, 60)) == binding.TG_ERR_INVALID_ARG      # lds < N
    assert call((8, 10)) == binding.TG_ERR_MISALIGNED       # ldq not a multiple of 4
    assert call((1, p + 4)) == binding.TG_ERR_MISALIGNED    # Wq not 16-byte aligned
    assert call((4, 0)) == binding.TG_OK                    # M == 0
    # plan options out of range are rejected before any device work
    for opts in ({"pair": 2}, {"pair": -2}, {"tail": 2}, {"tail": -2}, {"swap_ab": 3},
                 {"block_n": 192}, {"max_ctas": -1}, {"dequant_first": 2},
                 {"dequant_first": -2}):
        assert binding.tg_gemm_w4a16_f16(p, p, p, p, 64, 64, 64, 64, 8, 64, 64, 128,
                                         options=opts) == binding.TG_ERR_INVALID_ARG, opts


def test_plan_tail_split(lib):
    # by default: 1024 pair tiles on 76 clusters leave 36 for a last wave, run as 72 K halves
    p = _plan(8192, 8192, 8192)
    assert p["cta_pair"] == 1 and p["tail_tiles"] == 36 and p["units"] == 1024 + 36
    assert p["workspace_bytes"] >= 36 * 2 * 256 * 256 * 4
    assert _plan(8192, 8192, 8192, options={"tail": 1}) == p
    # 64 pair tiles on 76 clusters: no full wave before the last, nothing to balance
    assert _plan(2048, 2048, 2048)["tail_tiles"] == 0
    q = _plan(8192, 8192, 8192, options={"tail": -1})
    assert q["tail_tiles"] == 0 and q["units"] == 1024 and q["workspace_bytes"] == 0
    # no tail split when more than half the clusters would be busy, or with split-K
    assert _plan(300, 600, 1500, options={"pair": 1, "tail": 1, "max_ctas": 6})["tail_tiles"] == 0
    assert _plan(300, 600, 1500, options={"pair": 1, "tail": 1, "max_ctas": 8})["tail_tiles"] == 2
    assert _plan(8192, 8192, 8192, options={"split_k": 2, "tail": 1})["tail_tiles"] == 0


def test_noalloc_workspace_bound_cannot_overflow(lib):
    # The fixed-workspace entry point refuses, on the host and before any device work, every
    # problem whose split partials exceed its array.  Shapes near the 2^31 dimension limit make
    # splits * M * ldw * 4 exceed 2^64, which a plain product would wrap past the bound.
    big = (1 << 31) - 1024
    p = 4096
    cases = [
        (big, big, 64, 1),          # M * ldw * 4 ~ 2^64
        (big, 8, 64 * 8, 8),        # splits x a per-split slice just over 2^34
        (1, big, 64, 1),            # one row wider than the array
        (4096, 4096, 1024, 2),      # 128 MiB of partials against 64 MiB
    ]
    for M, N, K, split in cases:
        st = binding.tg_gemm_relu_f16_splitk_noalloc(p, p, p, M, N, K, -(-K // 8) * 8,
                                                     -(-N // 8) * 8, N, 1, split, 0)
        assert st == binding.TG_ERR_NO_WORKSPACE, (M, N, K, split, st)
    # argument errors come first, also without a device
    assert binding.tg_gemm_relu_f16_splitk_noalloc(p, p, p, 4, 4, 4, 8, 8, 4, 1, -1, 0) == \
        binding.TG_ERR_INVALID_ARG
    assert binding.tg_gemm_relu_f16_splitk_noalloc(p, p, p, 4, 4, 4, 8, 8, 3, 1, 1, 0) == \
        binding.TG_ERR_INVALID_ARG
