"""Parity of the fused epilogue C = fp16(act(A·B + bias) + residual) through the C ABI
(tg_gemm_f16_epilogue) with the oracle's float64 epilogue, on both kernels, on the direct
path (epilogue in the GEMM kernel) and on the split-K path (epilogue in the reduction)."""

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


ACT = {"none": 0, "relu": 1, "gelu": 2, "gelu_tanh": 3}


def run(a, b, act, bias=None, residual=None, options=None, ldc=None, inplace=False):
    M, K = a.shape
    N = b.shape[1]
    ldc = ldc or N
    A = torch.from_numpy(a).cuda()
    B = torch.from_numpy(b).cuda()
    C = torch.full((M, ldc), float("nan"), dtype=torch.float16, device="cuda")
    bias_t = torch.from_numpy(bias).cuda() if bias is not None else None
    res_t = None
    ldr = 0
    if residual is not None:
        if inplace:
            C[:, :N] = torch.from_numpy(residual).cuda()
            res_t, ldr = C, ldc
        else:
            res_t, ldr = torch.from_numpy(residual).cuda(), N
    st = binding.tg_gemm_f16_epilogue(
        A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, max(K, 1), N, ldc, ACT[act],
        bias_t.data_ptr() if bias_t is not None else 0,
        res_t.data_ptr() if res_t is not None else 0, ldr, options,
        torch.cuda.current_stream().cuda_stream)
    assert st == binding.TG_OK, binding.tg_status_string(st)
    torch.cuda.synchronize()
    out = C.cpu().numpy().view(np.uint16)
    return out[:, :N], out[:, N:]


def check(got, a, b, act, bias, residual):
    K = a.shape[1]
    r = oracle.gemm_epilogue(a, b, act, bias=bias, residual=residual)
    ref = {"out16_f64acc": r["out16_f64acc"], "acc_f64": r["pre_f64"]}
    zero_rule = act == "relu" and residual is None
    c = compare(got, ref, K, relu=zero_rule)
    assert c["out_of_tol"] == 0, c
    if zero_rule:
        assert c["zero_rule"] == 0 and c["negative_sign"] == 0, c
    return c


M, N, K = 333, 527, 1030


@pytest.mark.parametrize("act", list(ACT))
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("with_res", [False, True])
def test_epilogue_combinations_default_plan(act, with_bias, with_res):
    a = inputs.tensor(M, K, 51, 0)
    b = inputs.tensor(K, N, 51, 1)
    bias = (inputs.tensor(1, N, 52, 0).astype(np.float32) * 4).astype(np.float16).ravel() if with_bias else None
    res = inputs.tensor(M, N, 53, 1) if with_res else None
    got, pad = run(a, b, act, bias, res)
    check(got, a, b, act, bias, res)
    assert np.isnan(pad.view(np.float16)).all() if pad.size else True


@pytest.mark.parametrize("opts", [{"pair": 1}, {"pair": -1, "block_n": 192}, {"split_k": 3},
                                  {"pair": 1, "split_k": 2}, {"force_workspace": 1},
                                  {"pair": 1, "tail": 1, "max_ctas": 8}],
                         ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
@pytest.mark.parametrize("act", ["gelu", "relu"])
def test_epilogue_on_every_path(opts, act):
    a = inputs.tensor(M, K, 61, 0)
    b = inputs.tensor(K, N, 61, 1)
    bias = inputs.tensor(1, N, 62, 0).ravel()
    res = inputs.tensor(M, N, 63, 1)
    got, _ = run(a, b, act, bias, res, options=opts)
    check(got, a, b, act, bias, res)


def test_inplace_residual_and_odd_ldc():
    a = inputs.tensor(M, K, 71, 0)
    b = inputs.tensor(K, N, 71, 1)
    bias = inputs.tensor(1, N, 72, 0).ravel()
    res = inputs.tensor(M, N, 73, 1)
    for ldc in (N, 531, 536):
        got, pad = run(a, b, "gelu_tanh", bias, res, ldc=ldc, inplace=True)
        check(got, a, b, "gelu_tanh", bias, res)
        assert np.isnan(pad.view(np.float16)).all()


def test_k_zero_with_bias_and_residual():
    a = np.zeros((M, 0), np.float16)
    b = np.zeros((0, N), np.float16)
    bias = inputs.tensor(1, N, 81, 0).ravel()
    res = inputs.tensor(M, N, 82, 1)
    got, _ = run(a, b, "gelu", bias, res)
    r = oracle.gemm_epilogue(np.zeros((M, 1), np.float16), np.zeros((1, N), np.float16), "gelu",
                             bias=bias, residual=res)
    ref = {"out16_f64acc": r["out16_f64acc"], "acc_f64": r["pre_f64"]}
    assert compare(got, ref, 1, relu=False)["out_of_tol"] == 0
