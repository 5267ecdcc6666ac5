"""Pins for the oracle's blockwise Sylvester Hadamard rotation (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 7:
natural-order Sylvester H_128, normalised by 1/sqrt(128), applied blockwise
(H @ x per 128 rows, x @ H per 128 columns); decode order H_l -> x su -> H_r ->
x sv.  scipy.linalg.hadamard gives the same natural-order Sylvester matrix.
"""
import numpy as np
import pytest
from scipy.linalg import hadamard

import oracle

H = hadamard(128).astype(np.float64)


def _dense_forward(W, su, sv):
    W = W.astype(np.float64) * su[:, None] * sv[None, :]
    rows, cols = W.shape
    out = np.empty_like(W)
    for rb in range(0, rows, 128):
        for cb in range(0, cols, 128):
            out[rb:rb + 128, cb:cb + 128] = H @ W[rb:rb + 128, cb:cb + 128] @ H / 128.0
    return out


def test_basis_blocks_are_exact_outer_products():
    ones = np.ones(128, np.float32)
    for (i, j) in [(0, 0), (1, 0), (0, 5), (77, 3), (127, 127), (64, 31)]:
        E = np.zeros((128, 128), np.float32)
        E[i, j] = 1.0
        R = oracle.rotate_forward(E, ones, ones)
        want = np.outer(H[:, i], H[j, :]) / 128.0
        assert np.array_equal(R.astype(np.float64), want)


def test_unnormalised_transform_squares_to_128_identity():
    ones = np.ones(128, np.float32)
    for j in [0, 3, 100]:
        E = np.zeros((128, 128), np.float32)
        E[j, 0] = 1.0
        # forward twice: 2^-7 H (2^-7 H E H) H = 2^-14 * 128^2 E = E exactly
        R2 = oracle.rotate_forward(oracle.rotate_forward(E, ones, ones), ones, ones)
        assert np.array_equal(R2, E)


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384)])
def test_matches_dense_fp64_product(rows, cols):
    rng = np.random.default_rng(rows + cols)
    W = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    su = rng.choice([-1.0, 1.0], rows).astype(np.float32)
    sv = rng.choice([-1.0, 1.0], cols).astype(np.float32)
    R = oracle.rotate_forward(W, su, sv)
    ref = _dense_forward(W, su, sv)
    assert np.max(np.abs(R - ref)) <= 1e-6 * np.max(np.abs(ref))


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 256)])
def test_inverse_undoes_forward(rows, cols):
    rng = np.random.default_rng(3)
    W = rng.standard_normal((rows, cols)).astype(np.float32)
    su = rng.choice([-1.0, 1.0], rows).astype(np.float32)
    sv = rng.choice([-1.0, 1.0], cols).astype(np.float32)
    back = oracle.rotate_inverse(oracle.rotate_forward(W, su, sv), su, sv)
    assert np.max(np.abs(back - W)) <= 1e-5 * np.max(np.abs(W))
    # the inverse is su . (H Q H / 128) . sv in exact arithmetic
    Q = rng.standard_normal((rows, cols)).astype(np.float32)
    inv = oracle.rotate_inverse(Q, su, sv)
    ref = _dense_forward(Q, np.ones(rows), np.ones(cols)) * su[:, None] * sv[None, :]
    assert np.max(np.abs(inv - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_sign_vectors_apply_to_rows_and_columns():
    rng = np.random.default_rng(11)
    W = rng.standard_normal((128, 128)).astype(np.float32)
    su = np.ones(128, np.float32)
    sv = np.ones(128, np.float32)
    su[5] = -1.0
    sv[9] = -1.0
    A = oracle.rotate_forward(W, su, sv)
    W2 = W.copy()
    W2[5, :] *= -1
    W2[:, 9] *= -1
    B = oracle.rotate_forward(W2, np.ones(128, np.float32), np.ones(128, np.float32))
    assert np.max(np.abs(A - B)) <= 1e-6 * np.max(np.abs(B))
