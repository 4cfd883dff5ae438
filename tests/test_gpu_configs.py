"""Parity at the five named workloads' full sizes, in the launch configuration bench.py times
(the default plan through tg_gemm_relu_f16, natural leading dimensions).

Every output of every workload is compared with the oracle, element by element:
  - against the float64-accumulated result (authoritative): the tolerance
    |gpu - ref| <= 2 ulp16(ref) + 1e-4 sqrt(K) and the zero rule of tests/parity.py;
  - against the float32-accumulated result (the method's own arithmetic: a float32 fragment
    cleared, accumulated and passed through max(x, 0) before the fp16 copy, TileLang
    paper-reading page, section 2), with the same tolerance.
Integer-valued inputs of the same shapes make every partial sum exact in any order, so there
the whole output must equal the float32 oracle bit for bit, split-K and ragged edges included.
The output is also checked to be bitwise reproducible across two calls.

Per workload the test records the largest error in fp16 ulps, the relative Frobenius error,
the number of outputs equal to each reference bit for bit, the band count (|float64 sum| <
1e-4 sqrt(K), where no float32 kernel can decide the sign) and the literal zero-rule count
(nonzero outputs where the float64 sum is <= 0).  With TG_PARITY_REPORT set to a path, the
module writes them there as a markdown table."""

import os
import time

import numpy as np
import pytest

import oracle
from fp16_gemm_relu_gb300 import binding, inputs, workloads

from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

_REPORT = []


@pytest.fixture(scope="module", autouse=True)
def _built():
    from fp16_gemm_relu_gb300 import build

    build.build()
    torch.cuda.set_device(0)
    yield
    st, word = binding.tg_device_error_check(clear=True)
    assert st == binding.TG_OK, f"device error word {word:#x}"
    path = os.environ.get("TG_PARITY_REPORT")
    if path and _REPORT:
        with open(path, "w") as f:
            f.write(_report_markdown())


def _report_markdown():
    head = ("| workload | M x N x K | inputs | reference | outputs | out of tol | max ulp | "
            "max abs | rel. Frobenius | bitwise equal | band | zero rule (<= -tau) | "
            "literal zero rule (<= 0) | plan | oracle s |\n"
            "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|\n")
    rows = []
    for r in _REPORT:
        rows.append(
            f"| {r['workload']} | {r['shape']} | {r['inputs']} | {r['ref']} | {r['n']} | "
            f"{r['out_of_tol']} | {r['max_ulp_err']:.3g} | {r['max_abs_err']:.3g} | "
            f"{r['rel_fro']:.3g} | {r['bitwise_equal']} | {r.get('band', '-')} | "
            f"{r.get('zero_rule', '-')} | {r.get('literal_zero_rule', '-')} | {r['plan']} | "
            f"{r['oracle_s']:.1f} |")
    return head + "\n".join(rows) + "\n"


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
    C2 = torch.empty_like(C)
    st = binding.tg_gemm_relu_f16(A.data_ptr(), B.data_ptr(), C2.data_ptr(), M, N, K, K, N, N,
                                  binding.TG_EPILOGUE_RELU, torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16)), "not bitwise reproducible"
    del A, B, C2
    out = C.cpu().numpy().view(np.uint16)
    del C
    torch.cuda.empty_cache()
    return out


def _plan_text(M, N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = binding.tg_plan_query(0x1000, 0x2000, 0x3000, M, N, K, K, N, N, sms)
    assert st == binding.TG_OK
    kind = "pair 256x256" if p["cta_pair"] else f"128x{p['block_n']}"
    return f"{kind}, split {p['split_k']}, tail {p['tail_tiles']}"


def _record(wl, inputs_kind, c, oracle_s):
    r = dict(c)
    r.update(workload=wl.name, shape=f"{wl.M}x{wl.N}x{wl.K}", inputs=inputs_kind,
             plan=_plan_text(wl.M, wl.N, wl.K), oracle_s=oracle_s)
    _REPORT.append(r)
    print(r)


@pytest.mark.parametrize("name", workloads.ORDER)
def test_workload_full_parity(name):
    wl = workloads.get(name)
    a, b = wl.make_a(), wl.make_b()
    got = run_default(a, b)
    t0 = time.perf_counter()
    ref = oracle.gemm_relu(a, b, relu=True)
    dt = time.perf_counter() - t0
    del a, b
    c64 = assert_parity(got, ref, wl.K, True, where=f"{name} vs float64 oracle")
    _record(wl, "workload", c64, dt)
    c32 = assert_parity(got, ref, wl.K, True, where=f"{name} vs float32 oracle",
                        key="out16_f32acc")
    _record(wl, "workload", c32, dt)
    assert c64["rel_fro"] < 1e-3, c64  # fp16 output rounding alone is ~2e-4


@pytest.mark.parametrize("name", ["square2048", "square8192", "skinny64x28672x8192",
                                  "ragged4095x3073x65537"])
def test_workload_integer_inputs_bitwise(name):
    wl = workloads.get(name)
    a = inputs.tensor(wl.M, wl.K, wl.seed, 0, "int")
    b = inputs.tensor(wl.K, wl.N, wl.seed, 1, "int")
    got = run_default(a, b)
    t0 = time.perf_counter()
    ref = oracle.gemm_relu(a, b, relu=True, want=("f32",))
    dt = time.perf_counter() - t0
    c = assert_parity(got, {**ref, "out16_f64acc": ref["out16_f32acc"]}, wl.K, True,
                      where=f"{name} integer inputs", key="out16_f32acc")
    _record(wl, "integers in [-2, 2]", c, dt)
    np.testing.assert_array_equal(got, ref["out16_f32acc"])


def test_default_tail_split_with_ragged_edges():
    # 20 x 16 = 320 pair tiles: four full waves of 76 clusters, then 16 tiles that the default
    # plan runs as 32 K halves.  M, N and K all end in partial tiles (5000 = 19*256 + 136,
    # 4000 = 15*256 + 160, 1500 = 23*64 + 28), so the split tiles include edge tiles and the
    # second K half ends in a partial k-block.  (At K = 1000 the plan keeps 128 x 256 tiles.)
    M, N, K = 5000, 4000, 1500
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = binding.tg_plan_query(0x1000, 0x2000, 0x3000, M, N, K, K, N, N, sms)
    assert st == binding.TG_OK and plan["cta_pair"] == 1
    clusters = plan["grid"] // 2
    r = (plan["tiles_m"] * plan["tiles_n"]) % clusters
    assert plan["tail_tiles"] == (r if 0 < 2 * r <= clusters else 0)
    a = inputs.tensor(M, K, 61, 0)
    b = inputs.tensor(K, N, 61, 1)
    full = run_default(a, b)
    assert_parity(full, oracle.gemm_relu(a, b, relu=True), K, True, where="tail split, ragged")
    ai = inputs.tensor(M, K, 64, 0, "int")
    bi = inputs.tensor(K, N, 64, 1, "int")
    fi = run_default(ai, bi)
    refi = oracle.gemm_relu(ai, bi, relu=True, want=("f32",))
    np.testing.assert_array_equal(fi, refi["out16_f32acc"])
