"""Pins for the oracle's output-channel regularisation (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 8 and the
test list's test_regularize entry: block_rms accuracy and slice-boundary
accumulation, the skew heuristic in both directions, zero-channel flooring, the
all-zero flag, the round trip and non-mutation.
"""
import numpy as np
import pytest

import oracle
from oracle import regularize as OR


def test_block_rms_slice_order_hand_example():
    # rows = 128 -> 32 slices of 4 rows.  Column 0: row 0 holds 2^27 (square 2^54,
    # ulp 4), every other row 1.  Slice 0 adds three 1s to 2^54 one at a time
    # (each lost: 2^54 + 1 rounds back); slices 1..31 each sum to exactly 4, and
    # 2^54 + 4k is exact: total 2^54 + 124.  A plain running sum would give 2^54,
    # the exact sum is 2^54 + 127.
    W = np.ones((128, 2), dtype=np.float32)
    W[0, 0] = 2.0 ** 27
    S = OR.block_sumsq_cols(W)
    assert S[0] == 2.0 ** 54 + 124
    assert S[1] == 128.0


def test_block_rms_exact_on_integers_and_ragged_slices():
    rng = np.random.default_rng(1)
    for rows in (64, 100, 33, 7):       # 100 = 31 slices of 4 and an empty one; 7 < 32
        W = rng.integers(-50, 51, (rows, 9)).astype(np.float32)
        S = OR.block_sumsq_cols(W)
        want = (W.astype(np.int64) ** 2).sum(axis=0).astype(np.float64)
        assert np.array_equal(S, want)


def test_skew_both_directions_and_exact_values():
    k = 4096
    flat = np.full(k, 4.0)                             # d = 2 everywhere
    assert OR.skew(flat) == 81 / 4096                  # m = 4096 // 50 = 81, exact
    assert OR.regularize(np.ones((k, 16), np.float32), flat, np.ones(16))["apply_out"]
    spiky = np.full(k, 1.0)
    spiky[::50] = 10000.0                              # 82 channels with d = 100
    sk = OR.skew(spiky)
    assert sk == (81 * 100.0) / (82 * 100.0 + (k - 82))
    assert not OR.regularize(np.ones((k, 16), np.float32), spiky, np.ones(16))["apply_out"]
    assert OR.skew(np.zeros(k)) == 0.0


def test_zero_channels_floor_and_zero_flag():
    rng = np.random.default_rng(2)
    W = rng.standard_normal((256, 32)).astype(np.float32)
    W[:, [3, 17]] = 0.0
    sv = rng.choice([-1.0, 1.0], 32).astype(np.float32)
    r = OR.regularize(W, np.ones(256), sv)
    assert r["apply_out"] and not r["zeros"]
    assert r["sv_out"][3] == 0.0 and r["sv_out"][17] == 0.0
    assert not r["W_out"][:, [3, 17]].any()
    nz = [c for c in range(32) if c not in (3, 17)]
    assert np.all(np.sign(r["sv_out"][nz]) == sv[nz])
    z = OR.regularize(np.zeros((64, 16), np.float32), np.ones(64), np.ones(16))
    assert z["zeros"] and not z["sv_out"].any() and not z["W_out"].any()


@pytest.mark.parametrize("apply_out", [-1, 0, 1])
def test_round_trip_and_normalised_columns(apply_out):
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((512, 64)) * rng.uniform(0.01, 3.0, 64)).astype(np.float32)
    h = rng.uniform(0.5, 2.0, 512)
    sv = rng.choice([-1.0, 1.0], 64).astype(np.float32)
    W0, h0, sv0 = W.copy(), h.copy(), sv.copy()
    r = OR.regularize(W, h, sv, apply_out=apply_out)
    assert np.array_equal(W, W0) and np.array_equal(h, h0) and np.array_equal(sv, sv0)
    scale = np.abs(r["sv_out"]).astype(np.float64)
    back = r["W_out"].astype(np.float64) * scale[None, :]
    ulp = np.spacing(np.abs(W).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(back - W) <= ulp)
    exact_ss = (W.astype(np.float64) ** 2).sum(axis=0)
    if r["apply_out"]:
        col_rms = np.sqrt((r["W_out"].astype(np.float64) ** 2).mean(axis=0))
        assert np.all(np.abs(col_rms - 1.0) < 1e-6)
        assert np.allclose(scale, np.sqrt(exact_ss / 512), rtol=1e-6)
    else:
        g = np.sqrt(exact_ss.sum() / W.size)
        assert np.allclose(scale, g, rtol=1e-6)
        assert np.all(scale == scale[0])


def test_skew_sums_are_pairwise_trees():
    # d = (2^53, 1, 1, 1), m = 1.  Pairwise tree: (2^53 + 1) -> 2^53 (tie to even),
    # (1 + 1) = 2, then 2^53 + 2 exactly; a running sum would lose every 1 and give
    # 2^53 (skew exactly 1).
    h = np.array([2.0 ** 106, 1.0, 1.0, 1.0], dtype=np.float32)
    assert OR.skew(h) == 2.0 ** 53 / (2.0 ** 53 + 2.0)
