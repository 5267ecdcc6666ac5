"""Pins for the oracle's mul1 codebook and fp16 rounding (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 5: the mul1
codebook is procedural and its levels are fp16 values.  The multiplier and the
scale constant are this build's reading (the page gives neither); the tests
check the oracle against numpy's own byte view and IEEE float16 cast.
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle


def test_round_fp16_matches_numpy_float16_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 4,
        (rng.standard_normal(50000) * 1e-5).astype(np.float32),      # subnormal halves
        (rng.standard_normal(20000) * 7e4).astype(np.float32),       # overflow region
        np.float32([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -24,
                    2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11,
                    1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -11 + 2.0 ** -20]),
    ]).astype(np.float32)
    # exact halfway points between adjacent halves (ties must go to even)
    h = np.arange(0x3C00, 0x3E00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mid, -mid])
    ours = oracle.round_fp16(x)
    with np.errstate(over="ignore"):            # the overflow region rounds to +-inf by design
        ref = x.astype(np.float16).astype(np.float32)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def _bytesum_numpy(n_states):
    s = np.arange(n_states, dtype=np.uint64)
    x = ((s * np.uint64(oracle.mul1_multiplier())) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    return x.view(np.uint8).reshape(-1, 4).astype(np.int64).sum(axis=1)


def test_mul1_constant_is_inverse_bytesum_sd():
    b = _bytesum_numpy(65536)
    n = b.size
    s1, s2 = int(b.sum()), int((b * b).sum())
    getcontext().prec = 50
    var = Decimal(n * s2 - s1 * s1) / Decimal(n * n)
    c = Decimal(1) / var.sqrt()
    assert np.float32(float(c)) == np.float32(oracle.mul1_constant())


def test_mul1_table_matches_independent_numpy_evaluation():
    b = _bytesum_numpy(65536)
    c = np.float32(oracle.mul1_constant())
    ref = ((b - 510).astype(np.float32) * c).astype(np.float32).astype(np.float16).astype(np.float32)
    ours = oracle.mul1_table()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_mul1_table_properties():
    v = oracle.mul1_table().astype(np.float64)
    # every level is an fp16 value
    assert np.array_equal(v.astype(np.float16).astype(np.float64), v)
    # state 0 multiplies to 0: byte sum 0, the lowest level
    assert v[0] == float(np.float16(np.float32(-510) * np.float32(oracle.mul1_constant())))
    assert v[0] == v.min()
    # roughly standard: mean 0, sd within 1% of 1 (the scale was chosen for that)
    assert abs(v.mean()) < 0.01
    assert abs(v.std() - 1.0) < 0.01
    # the byte-sum levels of this multiplier: 913 distinct values
    assert len(np.unique(v)) == 913
    assert -3.5 < v.min() < -3.4 and 3.2 < v.max() < 3.4


def test_mul1_value_scalar_agrees_with_table():
    t = oracle.mul1_table()
    lib = oracle._load()
    for s in [0, 1, 2, 255, 256, 4095, 32767, 32768, 65534, 65535]:
        assert np.float32(lib.ora_mul1_value(s)) == t[s]
