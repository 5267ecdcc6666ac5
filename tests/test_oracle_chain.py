"""Pins for the oracle's decode of packed codes and its full evaluation chain
(not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 5 (states
are decoded to fp16 mul1 levels), item 7 (the decoded values are multiplied by
the scale before the inverse rotation, whose order is H_l -> x su -> H_r -> x
sv) and item 10 (reconstruction MSE against the original weight).  The
expected values are built here from pieces pinned elsewhere -- the mul1 table
(numpy byte-view evaluation), the state unpacking (hand-derived golden words),
scipy's Sylvester Hadamard matrix -- composed with numpy in binary64 or with
numpy's correctly rounded float32 product, so a misreading of the order (scale
applied as a multiply by 1/s, the level rounded after scaling, tiles placed
transposed, the MSE taken in the rotated domain, su and sv swapped) fails.
"""
import numpy as np
import pytest
from scipy.linalg import hadamard

import oracle
from exl3_trellis_weight_gb300 import inputs

H = hadamard(128).astype(np.float64)
SCALE = 0.0213   # not a power of two: fl(v * s) and fl(v * fl(1/s)) differ


def _block_h(X):
    """H_128 X H_128 per 128x128 block (binary64, unnormalised)."""
    out = np.empty_like(X)
    for rb in range(0, X.shape[0], 128):
        for cb in range(0, X.shape[1], 128):
            out[rb:rb + 128, cb:cb + 128] = H @ X[rb:rb + 128, cb:cb + 128] @ H
    return out


def test_decode_values_is_the_fp32_product_of_level_and_scale():
    rng = np.random.default_rng(5)
    states = rng.integers(0, 1 << 16, 4096).astype(np.uint32)
    table = oracle.mul1_table()
    got = oracle.decode_values(states, SCALE)
    want = table[states] * np.float32(SCALE)           # one correctly rounded fp32 product
    assert got.dtype == np.float32
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # the readings this excludes
    inv = np.float32(1.0) / np.float32(SCALE)
    times_inv = (table[states] / inv).astype(np.float32)
    assert not np.array_equal(got.view(np.uint32), times_inv.view(np.uint32))
    b = ((states.astype(np.uint64) * np.uint64(oracle.mul1_multiplier())) & np.uint64(0xFFFFFFFF))
    bytesum = b.astype(np.uint32).view(np.uint8).reshape(-1, 4).astype(np.int64).sum(axis=1)
    unrounded = (bytesum - 510).astype(np.float32) * np.float32(oracle.mul1_constant())
    rounded_after = (unrounded * np.float32(SCALE)).astype(np.float16).astype(np.float32)
    assert not np.array_equal(got.view(np.uint32), rounded_after.view(np.uint32))
    # a state's level at scale 1 is the table entry itself
    assert np.array_equal(oracle.decode_values(states, 1.0).view(np.uint32),
                          table[states].view(np.uint32))


@pytest.mark.parametrize("K", [2, 3])
def test_decode_matrix_places_tiles_row_major(K):
    rows, cols = 48, 80                              # 3 x 5 tiles: a transposition shows
    n = (rows // 16) * (cols // 16)
    rng = np.random.default_rng(10 + K)
    words = rng.integers(0, 1 << 16, (n, 16 * K)).astype(np.uint16)
    got = oracle.decode_matrix(words.reshape(rows // 16, cols // 16, 16 * K), rows, cols, K, SCALE)
    table = oracle.mul1_table()
    vals = np.stack([table[oracle.unpack_states(words[t], K)] for t in range(n)])
    vals = (vals * np.float32(SCALE)).astype(np.float32)
    want = vals.reshape(rows // 16, cols // 16, 16, 16).transpose(0, 2, 1, 3).reshape(rows, cols)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_evaluate_matrix_composition_against_dense_binary64():
    rows, cols, K, g = 256, 384, 2, 0.9
    Wb = inputs.linear_bf16(rows, cols, 61, 0.02)
    su, sv = (t.numpy() for t in inputs.sign_pair(rows, cols, 61))
    W = Wb.float().numpy()
    r = oracle.evaluate_matrix(W, su, sv, K, g)
    # forward rotation: 2^-7 H (su . W . sv) H per block
    R64 = _block_h(W.astype(np.float64) * su[:, None] * sv[None, :]) / 128.0
    assert np.max(np.abs(r["R"] - R64)) <= 1e-6 * np.max(np.abs(R64))
    # sigma = rms(R) in binary64, s = fl32(g sigma)
    sigma = np.sqrt(np.mean(r["R"].astype(np.float64) ** 2))
    assert abs(r["sigma"] - sigma) <= 1e-12 * sigma
    assert r["scale"] == float(np.float32(g * r["sigma"]))
    assert r["inv_scale"] == float(np.float32(1.0) / np.float32(r["scale"]))
    # the reconstruction decodes the codes at s (not 1/s)
    Yhat = oracle.decode_matrix(r["codes"], rows, cols, K, r["scale"])
    assert np.array_equal(r["Yhat"].view(np.uint32), Yhat.view(np.uint32))
    # inverse rotation: What = 2^-7 su . (H Yhat H) . sv
    What64 = _block_h(r["Yhat"].astype(np.float64)) / 128.0 * su[:, None] * sv[None, :]
    assert np.max(np.abs(r["What"] - What64)) <= 1e-6 * np.max(np.abs(What64))
    swapped = _block_h(r["Yhat"].astype(np.float64) * su[:, None] * sv[None, :]) / 128.0
    assert np.max(np.abs(r["What"] - swapped)) > 1e-3 * np.max(np.abs(What64))
    # MSE in the weight domain, against W (not R)
    mse = np.mean((W.astype(np.float64) - r["What"].astype(np.float64)) ** 2)
    assert abs(r["mse"] - mse) <= 1e-12 * mse
    # the rotation is orthogonal, so the rotated-domain MSE agrees to rounding
    # only; that rounding (about 1e-10 relative here) is far outside the 1e-12
    # above, so an oracle that measured in the rotated domain fails the check
    mse_rot = np.mean((r["R"].astype(np.float64) - r["Yhat"].astype(np.float64)) ** 2)
    assert 1e-11 * mse < abs(mse_rot - r["mse"]) < 1e-6 * mse
