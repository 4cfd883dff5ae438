"""Comparison of the CUDA path's fp16 output with the oracle.

Tolerance (stated for the method's fp32-accumulate / fp16-output arithmetic):
    |gpu - ref| <= 2 * ulp16(ref) + 1e-4 * sqrt(K)
where ref is the oracle's float64-accumulated result rounded once to fp16 and ulp16(r) is
2^(floor(log2|r|) - 10) for |r| >= 2^-14, else 2^-24.  The kernel sums in a blocked order, so
its float32 sum can differ from the oracle's by a few float32 rounding errors; after rounding
to fp16 that is at most one fp16 ulp apart, well inside the bound.

Zero rule (relu epilogue): every element whose float64 pre-activation sum is <= -tau,
tau = 1e-4 * sqrt(K), must be exactly +0 (0x0000); elements with |sum| < tau may round either
way, so there the output must only be non-negative (sign bit clear) and within tolerance.
The count of outputs that are nonzero where the float64 sum is <= 0 is reported.
"""

from __future__ import annotations

import numpy as np

import oracle


def ulp16(r: np.ndarray) -> np.ndarray:
    a = np.abs(r)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.where(a >= 2.0 ** -14, 2.0 ** (e - 10), 2.0 ** -24)


def compare(got_bits: np.ndarray, ref: dict, K: int, relu: bool = True) -> dict:
    """got_bits: uint16 GPU output; ref: oracle.gemm_relu(...) result with the f64 keys."""
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    r = oracle.f16_bits_to_f64(ref["out16_f64acc"])
    g = oracle.f16_bits_to_f64(got_bits)
    pre = ref["acc_f64"]
    tau = 1e-4 * np.sqrt(max(K, 1))
    tol = 2.0 * ulp16(r) + tau
    inf = np.isinf(r)
    err = np.where(inf, np.where(g == r, 0.0, np.inf), np.abs(g - r))
    out = {
        "n": int(got_bits.size),
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "max_ulp_err": float((err / ulp16(r)).max()) if err.size else 0.0,
        "out_of_tol": int((err > tol).sum()),
        "rel_fro": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)) if err.size else 0.0,
    }
    if relu:
        out["negative_sign"] = int(((got_bits & 0x8000) != 0).sum())
        out["zero_rule"] = int(((pre <= -tau) & (got_bits != 0)).sum())
        out["literal_zero_rule"] = int(((pre <= 0) & (got_bits != 0)).sum())
        out["band"] = int((np.abs(pre) < tau).sum())
    return out


def assert_parity(got_bits, ref, K, relu=True, where=""):
    c = compare(got_bits, ref, K, relu)
    ok = c["out_of_tol"] == 0 and (not relu or (c["zero_rule"] == 0 and c["negative_sign"] == 0))
    assert ok, f"parity failed {where}: {c}"
    return c
