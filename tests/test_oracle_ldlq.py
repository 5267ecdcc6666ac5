"""Pins for the oracle's block LDL and LDLQ error feedback (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 3 and the
test list's test_ldlq / test_ldlq_loop entries: L L^T = H, the block-diagonal
inversion fold with identity diagonal blocks, the damping retry schedule on
ill-conditioned Hessians, identity-factor equivalence with independent tile
quantisation, exact additive target correction, a dense transcription, and the
objective improvement on a correlated Hessian.
"""
import numpy as np
import pytest
import scipy.linalg

import oracle
from oracle import ldlq as O
from exl3_trellis_weight_gb300 import inputs


def _int_factor(n, seed):
    """Integer lower-triangular factor with power-of-two diagonal: H = L L^T is
    exact in binary64 and so is every step of the textbook Cholesky."""
    rng = np.random.default_rng(seed)
    L = np.tril(rng.integers(-3, 4, (n, n)), -1).astype(np.float64)
    L[np.diag_indices(n)] = rng.choice([1.0, 2.0, 4.0], n)
    return L, L @ L.T


def test_cholesky_exact_on_integer_factor():
    L, H = _int_factor(48, 1)
    Lo, rc = O.cholesky(H)
    assert rc == 0
    assert np.array_equal(Lo, L)


def test_cholesky_matches_lapack_and_reconstructs():
    H = inputs.spd_hessian(128, 3).numpy()
    Lo, rc = O.cholesky(H)
    assert rc == 0
    Ln = np.linalg.cholesky(H)
    assert np.max(np.abs(Lo - Ln)) <= 1e-10 * np.max(np.abs(Ln))
    assert np.max(np.abs(Lo @ Lo.T - H)) <= 1e-12 * np.max(np.abs(H))
    assert np.all(np.triu(Lo, 1) == 0)


def test_cholesky_reports_first_bad_pivot():
    H = np.eye(32)
    H[5, 5] = -1.0
    assert O.cholesky(H)[1] == 6
    H = np.eye(32)
    H[0, 0] = 0.0
    assert O.cholesky(H)[1] == 1
    # 2x2 leading block [[1, 2], [2, 1]] is indefinite: the second pivot is 1 - 4 < 0
    H = np.eye(32)
    H[0, 1] = H[1, 0] = 2.0
    assert O.cholesky(H)[1] == 2


@pytest.mark.parametrize("need", [0, 1, 3, 10])
def test_damping_retry_count(need):
    n = 64
    eigs = np.linspace(0.5, 2.0, n)
    delta = 2 * O.SIGMA_REG * eigs.mean()          # 2 sigma_reg mean(diag H)
    if need > 0:
        # smallest eigenvalue placed half a step below the need-th damping level
        eigs[0] = -(need - 0.5) * delta
        delta = 2 * O.SIGMA_REG * eigs.mean()
        eigs[0] = -(need - 0.5) * delta
    H = inputs.spectral_hessian(n, eigs, seed=5).numpy()
    M, a, _ = O.block_ldl(H)
    assert a == need


def test_damping_gives_up_after_ten_retries():
    n = 64
    eigs = np.linspace(0.5, 2.0, n)
    eigs[0] = -1.0                                   # needs ~40 damping steps
    H = inputs.spectral_hessian(n, eigs, seed=6).numpy()
    M, a, _ = O.block_ldl(H)
    assert a == -1 and M is None
    assert O.block_ldl(H, max_retries=60)[1] > 10


def test_block_fold_exact_on_dyadic_factor():
    n = 48
    L, H = _int_factor(n, 2)
    M, a, Lo = O.block_ldl(H)
    assert a == 0 and np.array_equal(Lo, L)
    want = np.zeros((n, n))
    for b in range(n // 16):
        cs = slice(16 * b, 16 * b + 16)
        X = scipy.linalg.solve_triangular(L[cs, cs], np.eye(16), lower=True)
        want[16 * (b + 1):, cs] = L[16 * (b + 1):, cs] @ X
    assert np.array_equal(M.astype(np.float64), want.astype(np.float32).astype(np.float64))
    # diagonal blocks (identity in M) and the upper part are stored as zero
    for b in range(n // 16):
        assert not M[16 * b:16 * b + 16, 16 * b:].any()


def test_block_fold_factorises_hessian():
    n = 128
    H = inputs.spd_hessian(n, 4).numpy()
    M32, a, L = O.block_ldl(H)
    assert a == 0
    Mf = M32.astype(np.float64) + np.eye(n)          # add back the identity blocks
    Lam = np.zeros((n, n))
    for b in range(n // 16):
        cs = slice(16 * b, 16 * b + 16)
        Lam[cs, cs] = L[cs, cs]
    assert np.max(np.abs(Mf @ Lam - L)) <= 1e-6 * np.max(np.abs(L))
    D = Lam @ Lam.T
    assert np.max(np.abs(Mf @ D @ Mf.T - H)) <= 1e-5 * np.max(np.abs(H))


def _dyadic_case(n, cols, seed):
    rng = np.random.default_rng(seed)
    R = (rng.integers(-16, 17, (n, cols)) / 8.0).astype(np.float32)
    M = np.zeros((n, n), dtype=np.float32)
    for b in range(n // 16):
        lo = 16 * (b + 1)
        M[lo:, 16 * b:16 * b + 16] = rng.choice([0.0, 0.5, -0.5], (n - lo, 16))
    return R, M


@pytest.mark.parametrize("n", [32, 48])
def test_ldlq_additive_correction_exact(n):
    # dyadic data at scale 1: every product, partial sum and the target add are
    # exact in fp32, so the targets equal the binary64 dense expression exactly
    R, M = _dyadic_case(n, 32, 11 + n)
    res = O.ldlq(R, M, 2, 1.0, threads=1)
    E = R.astype(np.float64) - res["Q"].astype(np.float64)
    for b in range(n // 16):
        rs = slice(16 * b, 16 * b + 16)
        below = slice(16 * (b + 1), n)
        want = R[rs].astype(np.float64) + M[below, rs].astype(np.float64).T @ E[below]
        assert np.array_equal(res["U"][rs].astype(np.float64), want)


def test_ldlq_identity_factor_equals_plain_quantisation():
    n, cols = 64, 48
    R = inputs.iid_f32(n, cols, 21).numpy()
    M = np.zeros((n, n), dtype=np.float32)            # block-diagonal Hessian
    s = np.float32(oracle.rms(R))
    res = O.ldlq(R, M, 3, float(s))
    st, _ = oracle.encode_matrix(R, 3, float(np.float32(1.0) / s))
    assert np.array_equal(res["states"], st)
    assert np.array_equal(res["U"], R)


def test_ldlq_dense_transcription_and_bottom_span():
    n, cols, K = 96, 64, 2
    H = inputs.spd_hessian(n, 7, rho=0.95).numpy()
    M, a, _ = O.block_ldl(H)
    R = inputs.iid_f32(n, cols, 8).numpy()
    s = float(np.float32(oracle.rms(R)))
    res = O.ldlq(R, M, K, s)
    E = R.astype(np.float64) - res["Q"].astype(np.float64)
    Md = M.astype(np.float64)
    for b in range(n // 16):
        rs = slice(16 * b, 16 * b + 16)
        below = slice(16 * (b + 1), n)
        dense = R[rs].astype(np.float64) + Md[below, rs].T @ E[below]
        bound = 1e-6 * (1.0 + np.abs(Md[below, rs]).T @ np.abs(E[below]))
        assert np.all(np.abs(res["U"][rs] - dense) <= bound)
    # the bottom span has nothing below it: plain quantisation of R's last rows
    st, _ = oracle.encode_matrix(R[n - 16:], K, float(np.float32(1.0) / np.float32(s)))
    TC = cols // 16
    assert np.array_equal(res["states"][(n // 16 - 1) * TC:], st)


def test_ldlq_lowers_the_proxy_loss_on_a_correlated_hessian():
    n, cols, K = 256, 128, 2
    H = inputs.spd_hessian(n, 9, rho=0.95).numpy()
    M, a, _ = O.block_ldl(H)
    R = inputs.iid_f32(n, cols, 10).numpy()
    s = float(np.float32(oracle.rms(R)))
    res = O.ldlq(R, M, K, s)
    plain = np.zeros((n, n), dtype=np.float32)
    base = O.ldlq(R, plain, K, s)
    l_ldlq = O.proxy_loss(R, res["Q"], H)
    l_base = O.proxy_loss(R, base["Q"], H)
    assert l_ldlq < 0.8 * l_base
