"""Pins of the oracle's rotary position encoding (oracle.rope).

Each pin is fixed by the mathematics of a rotation by position-proportional angles,
not by re-typing the formula: the worked value of a 4-dim vector, identity at position
0, the norm of every rotated pair, composition of two rotations, and the property the
encoding exists for -- the score of a rotated query and key depends only on their
distance. A pair taken as adjacent dims, a wrong frequency exponent or a swapped sign
fails one of them.
"""

import numpy as np
import pytest

import oracle
from workloads import gen_queries, make_rng

D = 64


def test_worked_value_four_dims():
    # theta = (1, 10000^-1/2 = 0.01); x = e0 at position 1 -> (cos 1, 0, sin 1, 0)
    x = np.zeros((1, 1, 2, 4))
    x[0, 0, 0, 0] = 1.0
    x[0, 0, 1, 1] = 1.0  # second token: e1, at position 2 -> angle 2 * 0.01
    y = oracle.rope(x, "f64", np.array([1], np.int32))
    assert np.allclose(y[0, 0, 0], [np.cos(1.0), 0.0, np.sin(1.0), 0.0], atol=1e-15)
    assert np.allclose(y[0, 0, 1], [0.0, np.cos(0.02), 0.0, np.sin(0.02)], atol=1e-15)


def test_position_zero_is_the_identity():
    x = np.random.default_rng(1).standard_normal((2, 3, 1, D))
    y = oracle.rope(x, "f64", np.zeros(2, np.int32))
    assert np.array_equal(y, x)


def test_pairs_keep_their_norm():
    x = np.random.default_rng(2).standard_normal((2, 2, 5, D))
    y = oracle.rope(x, "f64", np.array([17, 3000], np.int32))
    n_in = x[..., : D // 2] ** 2 + x[..., D // 2:] ** 2
    n_out = y[..., : D // 2] ** 2 + y[..., D // 2:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12)
    assert not np.allclose(y, x)


def test_two_rotations_compose():
    x = np.random.default_rng(3).standard_normal((1, 2, 1, D))
    once = oracle.rope(oracle.rope(x, "f64", np.array([40], np.int32)), "f64",
                       np.array([2], np.int32))
    direct = oracle.rope(x, "f64", np.array([42], np.int32))
    assert np.allclose(once, direct, atol=1e-12)


@pytest.mark.parametrize("base", [10000.0, 500000.0])
def test_scores_depend_only_on_distance(base):
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, 1, D))
    k = rng.standard_normal((1, 1, 1, D))

    def score(m, n):
        qm = oracle.rope(q, "f64", np.array([m], np.int32), base)
        kn = oracle.rope(k, "f64", np.array([n], np.int32), base)
        return float(np.sum(qm * kn))

    for m, n in [(5, 2), (100, 0), (2047, 1500)]:
        s = score(m, n)
        for shift in (1, 13, 700):
            assert abs(score(m + shift, n + shift) - s) < 1e-9 * (1 + abs(s))
    assert abs(score(5, 2) - score(5, 3)) > 1e-6  # but it does depend on the distance


def test_16_bit_inputs_decode_exactly():
    # fp16/bf16 bits are decoded exactly, so the result equals the f64 path on the
    # decoded values
    rng = make_rng(5)
    for dtype in ("f16", "bf16"):
        x = gen_queries(rng, 2, 3, 4, D, dtype, 0.5)
        y16 = oracle.rope(x, dtype, np.array([0, 9], np.int32))
        y64 = oracle.rope(oracle.decode(x, dtype), "f64", np.array([0, 9], np.int32))
        assert np.array_equal(y16, y64)
