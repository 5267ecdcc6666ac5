"""Block LDL factorisation and LDLQ error feedback (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the page "EXL3 Intel Arc Quantizer", Core Implemented Architecture
item 3 ("Block LDLQ Decomposition & Preprocessing"): a Cholesky factor of the
Hessian with the inverse of its 16x16 block diagonal folded in,
M = L * blockdiag(L_bb)^-1, diagonal damping of 2 * sigma_reg * mean(diag H)
retried up to 10 times, and one-sided error feedback that walks the weight's
16-row spans bottom-up, adding to each span's targets the errors of the spans
already quantised, weighted by the strictly lower part of M.  The page states
no more than that; the readings below fill in the rest, each a choice made
where the page is silent:

  * weights are R [n, cols] (rows = input channels, the Hessian's index), the
    Hessian H [n, n] is symmetric positive definite in the same basis;
  * retry a (a = 0 .. max_retries) factors H + a * delta * I with
    delta = 2 * sigma_reg * mean(diag H), sigma_reg = 0.01 by default (the
    page's Hessian damping constant);
  * the proxy objective tr(E^T H E), E = R - Q, is minimised span by span:
    with H = M D M^T, span b's targets are
        U_b = fl32(R_b + sum_{i >= 16 (b + 1)} M[i, b-rows]^T E_i),
    the sum an fp32 fused-multiply-add chain over i from n - 1 down (the
    order in which rows are quantised), E_i = fl32(R_i - Q_i) in fp32;
  * each span is coded as 16x16 tiles at one scale s (codes from
    fl32(U * fl32(1 / s)), reconstruction Q = fl32(v * s)).

The arithmetic is in exl3_oracle.c (ora_cholesky, ora_cholesky_damped,
ora_block_fold, ora_ldlq_feedback); this module strings the steps together.
"""
from __future__ import annotations

import numpy as np

SIGMA_REG = 0.01
MAX_RETRIES = 10


def cholesky(H, diag_add: float = 0.0):
    """Textbook fp64 Cholesky; returns (L, failed_column or 0)."""
    import oracle
    from oracle import _load, _p
    H = np.ascontiguousarray(H, dtype=np.float64)
    n = H.shape[0]
    L = np.empty((n, n), dtype=np.float64)
    rc = _load().ora_cholesky(_p(H), n, float(diag_add), _p(L))
    return L, int(rc)


def block_ldl(H, sigma_reg: float = SIGMA_REG, max_retries: int = MAX_RETRIES):
    """Returns (M32 [n, n] float32, retries, L [n, n] float64); retries = -1 and
    M32 = None when every attempt failed."""
    from oracle import _load, _p
    H = np.ascontiguousarray(H, dtype=np.float64)
    n = H.shape[0]
    assert H.shape == (n, n) and n % 16 == 0
    L = np.empty((n, n), dtype=np.float64)
    lib = _load()
    a = int(lib.ora_cholesky_damped(_p(H), n, float(sigma_reg), int(max_retries), _p(L)))
    if a < 0:
        return None, -1, None
    M = np.empty((n, n), dtype=np.float32)
    lib.ora_block_fold(_p(L), n, _p(M))
    return M, a, L


def ldlq(R, M, K: int, scale: float, threads: int | None = None):
    """LDLQ of R [n, cols] with the folded factor M [n, n] at scale s.

    Returns dict(states [n/16 * cols/16, 256] uint32 in row-major tile order,
    codes [n/16, cols/16, 16K] uint16, Q [n, cols] float32, U [n, cols] float32
    (the targets each span was coded from)).
    """
    import oracle
    from oracle import _load, _p
    R = np.ascontiguousarray(R, dtype=np.float32)
    M = np.ascontiguousarray(M, dtype=np.float32)
    n, cols = R.shape
    assert n % 16 == 0 and cols % 16 == 0 and M.shape == (n, n)
    s = np.float32(scale)
    inv = np.float32(1.0) / s
    B, TC = n // 16, cols // 16
    acc = np.zeros((n, cols), dtype=np.float32)
    U = np.empty((n, cols), dtype=np.float32)
    Q = np.empty((n, cols), dtype=np.float32)
    states = np.empty((B * TC, 256), dtype=np.uint32)
    lib = _load()
    for j in range(B - 1, -1, -1):
        rs = slice(16 * j, 16 * j + 16)
        U[rs] = R[rs] + acc[rs]                       # fp32 add, one rounding
        st, _ = oracle.encode_matrix(U[rs], K, float(inv), threads=threads)
        states[j * TC:(j + 1) * TC] = st
        for t in range(TC):
            Q[rs, 16 * t:16 * t + 16] = oracle.decode_values(st[t], float(s)).reshape(16, 16)
        E = np.ascontiguousarray(R[rs] - Q[rs])       # fp32 subtract, one rounding
        if j > 0:
            lib.ora_ldlq_feedback(_p(acc), _p(M), n, cols, j, _p(E))
    codes = oracle.codes_from_states(states, n, cols, K)
    return dict(states=states, codes=codes, Q=Q, U=U)


def proxy_loss(R, Q, H) -> float:
    """tr(E^T H E) with E = R - Q, in binary64 (item 10's Hessian-weighted loss)."""
    E = np.asarray(R, dtype=np.float64) - np.asarray(Q, dtype=np.float64)
    return float(np.sum((np.asarray(H, dtype=np.float64) @ E) * E))
