"""The named relu(A·B) workloads: shapes, seeds and value distributions.

A is (M, K) and B is (K, N), both row-major fp16 with natural leading dimensions
(lda = K, ldb = N, ldc = N).  Inputs come from :mod:`fp16_gemm_relu_gb300.inputs`.
The 2048^3 shape with 128x128x32 tiles is the example GEMM of the TileLang practitioner
page (section 3.2); the rest span the compute-bound, memory-bound and ragged regimes.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import inputs


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    dist_a: str
    dist_b: str
    scale_a: float
    scale_b: float
    regime: str

    @property
    def lda(self) -> int:
        return self.K

    @property
    def ldb(self) -> int:
        return self.N

    @property
    def ldc(self) -> int:
        return self.N

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """Each operand read once and C written once, fp16."""
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)

    def make_a(self) -> np.ndarray:
        return inputs.tensor(self.M, self.K, self.seed, inputs.TENSOR_A, self.dist_a, self.scale_a)

    def make_b(self) -> np.ndarray:
        return inputs.tensor(self.K, self.N, self.seed, inputs.TENSOR_B, self.dist_b, self.scale_b)


def _wl(name, M, N, K, seed, dist_a="uniform", dist_b="uniform", scale_a=1.0, scale_b=1.0,
        regime="tensor"):
    return Workload(name, M, N, K, seed, dist_a, dist_b, scale_a, scale_b, regime)


WORKLOADS = {
    w.name: w
    for w in [
        _wl("square256", 256, 256, 256, 0, regime="launch"),
        _wl("square2048", 2048, 2048, 2048, 1),
        _wl("square8192", 8192, 8192, 8192, 2),
        _wl("skinny64x28672x8192", 64, 28672, 8192, 3, dist_a="normal", dist_b="normal",
            scale_b=1.0 / math.sqrt(8192), regime="hbm"),
        _wl("ragged4095x3073x65537", 4095, 3073, 65537, 4,
            scale_a=1.0 / math.sqrt(65537), scale_b=1.0 / math.sqrt(65537)),
    ]
}

ORDER = list(WORKLOADS)


def get(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {', '.join(ORDER)}") from None
