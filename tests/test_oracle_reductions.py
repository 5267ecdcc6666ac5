"""Pins for the oracle's fixed-order fp64 reductions (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 10
(reconstruction MSE).  The order is this build's reading: per 16x16 tile a
sequential row-major sum, then a pairwise tree over tiles.
"""
import math

import numpy as np

import oracle


def test_tree_sum_order_worked_example():
    # pairwise: (1 + 1e16) + (-1e16 + 1) = 1e16 - 1e16 = 0 ; sequential gives 1
    assert oracle.tree_sum(np.array([1.0, 1e16, -1e16, 1.0])) == 0.0
    # odd count: the last element moves up: ((a+b) + c)
    assert oracle.tree_sum(np.array([1e16, 1.0, 1.0])) == (1e16 + 1.0) + 1.0
    # five: ((a+b)+(c+d)) + e
    v = np.array([1.0, 2.0, 3.0, 4.0, 5.0])
    assert oracle.tree_sum(v) == 15.0
    assert oracle.tree_sum(np.array([])) == 0.0
    assert oracle.tree_sum(np.array([7.5])) == 7.5


def test_tree_sum_within_rounding_bound_of_exact_sum():
    rng = np.random.default_rng(0)
    for n in [1, 2, 3, 17, 1000, 65536, 100001]:
        v = rng.standard_normal(n) ** 2
        exact = math.fsum(v)
        depth = max(1, math.ceil(math.log2(n)))
        assert abs(oracle.tree_sum(v) - exact) <= depth * 2.3e-16 * math.fsum(np.abs(v))


def test_tile_sumsq_exact_on_small_integers():
    rng = np.random.default_rng(1)
    x = rng.integers(-50, 50, (64, 48)).astype(np.float32)
    r = rng.integers(-50, 50, (64, 48)).astype(np.float32)
    ts = oracle.tile_sumsq(x, r)
    d = (x.astype(np.int64) - r.astype(np.int64)) ** 2
    want = d.reshape(4, 16, 3, 16).sum(axis=(1, 3)).reshape(-1)
    assert np.array_equal(ts, want.astype(np.float64))
    ts0 = oracle.tile_sumsq(x)
    want0 = (x.astype(np.int64) ** 2).reshape(4, 16, 3, 16).sum(axis=(1, 3)).reshape(-1)
    assert np.array_equal(ts0, want0.astype(np.float64))


def test_rms_and_mse_definitions():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((128, 256)).astype(np.float32)
    assert abs(oracle.rms(x) - math.sqrt(math.fsum(x.astype(np.float64).ravel() ** 2) / x.size)) < 1e-12
    xi = rng.integers(-1000, 1000, (128, 256)).astype(np.float32)
    assert oracle.mse(xi, xi + np.float32(0.5)) == 0.25   # exact: integers + 0.5


def test_scale_for_rounds_product_then_reciprocal():
    s, inv = oracle.scale_for(1.25, 0.0123456789)
    assert s == float(np.float32(1.25 * 0.0123456789))
    assert inv == float(np.float32(1.0) / np.float32(s))
