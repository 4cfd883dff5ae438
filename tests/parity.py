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


def compare(got_bits: np.ndarray, ref: dict, K: int, relu: bool = True,
            key: str = "out16_f64acc") -> dict:
    """got_bits: uint16 GPU output; ref: an oracle.gemm_relu(...) result.  `key` names the
    reference the tolerance is measured against: the float64-accumulated result (authoritative)
    or "out16_f32acc", the float32-accumulated one (the method's own arithmetic).  The zero rule
    always uses the float64 pre-activation sum when the result holds it."""
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    ref_bits = ref[key]
    r = oracle.f16_bits_to_f64(ref_bits)
    g = oracle.f16_bits_to_f64(got_bits)
    tau = 1e-4 * np.sqrt(max(K, 1))
    u = ulp16(r)
    tol = 2.0 * u + tau
    inf = np.isinf(r)
    err = np.where(inf, np.where(g == r, 0.0, np.inf), np.abs(g - r))
    out = {
        "ref": key,
        "n": int(got_bits.size),
        "max_abs_err": float(err.max()) if err.size else 0.0,
        "max_ulp_err": float((err / u).max()) if err.size else 0.0,
        "out_of_tol": int((err > tol).sum()),
        "rel_fro": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)) if err.size else 0.0,
        "bitwise_equal": int((got_bits == ref_bits).sum()),
    }
    if relu:
        pre = ref["acc_f64"] if "acc_f64" in ref else ref["acc_f32"].astype(np.float64)
        out["negative_sign"] = int(((got_bits & 0x8000) != 0).sum())
        out["zero_rule"] = int(((pre <= -tau) & (got_bits != 0)).sum())
        out["literal_zero_rule"] = int(((pre <= 0) & (got_bits != 0)).sum())
        out["band"] = int((np.abs(pre) < tau).sum())
    return out


def assert_parity(got_bits, ref, K, relu=True, where="", key="out16_f64acc"):
    c = compare(got_bits, ref, K, relu, key)
    ok = c["out_of_tol"] == 0 and (not relu or (c["zero_rule"] == 0 and c["negative_sign"] == 0))
    assert ok, f"parity failed {where}: {c}"
    return c
