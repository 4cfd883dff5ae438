"""The seeded generator: published SplitMix64 outputs, determinism, ranges and moments."""

import numpy as np

from fp16_gemm_relu_gb300 import inputs, workloads


def test_splitmix64_known_answers():
    # SplitMix64 with initial state 0: the first outputs of the published reference generator
    x = inputs.raw_u64(np.uint64(0), 0, 3)
    assert [hex(int(v)) for v in x] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4",
                                       "0x6c45d188009454f"]


def test_counter_based_slices_agree():
    k = inputs.stream_key(9, 1, 0)
    whole = inputs.raw_u64(k, 0, 1000)
    np.testing.assert_array_equal(whole[400:700], inputs.raw_u64(k, 400, 300))


def test_deterministic_and_seed_dependent():
    a1 = inputs.tensor(64, 80, 3, 0)
    a2 = inputs.tensor(64, 80, 3, 0)
    b = inputs.tensor(64, 80, 3, 1)
    c = inputs.tensor(64, 80, 4, 0)
    np.testing.assert_array_equal(a1.view(np.uint16), a2.view(np.uint16))
    assert (a1 != b).mean() > 0.9 and (a1 != c).mean() > 0.9


def test_element_values_do_not_depend_on_shape_split():
    # element (r, c) is stream element r*cols + c: a (2, 50) tensor is a reshaped (1, 100) one
    x = inputs.tensor(2, 50, 8, 0)
    y = inputs.tensor(1, 100, 8, 0)
    np.testing.assert_array_equal(x.ravel().view(np.uint16), y.ravel().view(np.uint16))


def test_uniform_range_and_moments():
    x = inputs.tensor(512, 512, 1, 0).astype(np.float64)
    assert x.min() >= -1.0 and x.max() <= 1.0
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0 / 3.0) < 0.01


def test_normal_moments():
    x = inputs.tensor(512, 512, 3, 0, "normal").astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.02
    assert abs(((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3.0) < 0.1


def test_int_values():
    x = inputs.tensor(100, 100, 5, 0, "int")
    assert set(np.unique(x.astype(np.int64)).tolist()) == {-2, -1, 0, 1, 2}


def test_workloads_table():
    assert workloads.ORDER == ["square256", "square2048", "square8192", "skinny64x28672x8192",
                               "ragged4095x3073x65537"]
    w = workloads.get("ragged4095x3073x65537")
    assert (w.M, w.N, w.K, w.seed) == (4095, 3073, 65537, 4)
    assert w.flops == 2 * 4095 * 3073 * 65537
    s = workloads.get("skinny64x28672x8192")
    b = inputs.tensor(256, 64, s.seed, 1, s.dist_b, s.scale_b).astype(np.float64)
    assert abs(b.std() * np.sqrt(8192) - 1.0) < 0.05
