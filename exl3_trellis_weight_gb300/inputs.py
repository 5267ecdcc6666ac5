"""Seeded synthetic inputs for tests and benchmarks.

This module draws random numbers only; it holds none of the encoder's
arithmetic.  Both the CUDA path and the CPU oracle are fed the very same
tensors produced here (generated on the host with a seeded
``torch.Generator``), so a comparison never depends on how either side draws.

Workload shapes (weight matrices of a 4096-hidden decoder layer with 32 query
heads, 8 KV heads and a 12288-wide MLP):
  * ``iid_f32``       -- fp32 N(0, 1), used as already-rotated targets.
  * ``linear_bf16``   -- bf16 N(0, std^2), optionally with a fraction of
                         entries (chosen uniformly without replacement)
                         multiplied by an outlier factor.
  * ``student_t_bf16``-- bf16 Student-t (nu degrees of freedom) scaled to a
                         target standard deviation; t = z / sqrt(chi2_nu / nu)
                         with chi2_nu a sum of nu squared standard normals.
  * ``signs``         -- fp32 vector of independent +-1 with probability 1/2.
  * ``spd_hessian``   -- fp64 [n, n] stand-in for a harvested input Hessian:
                         H = X^T X / N + 0.01 mean(diag) I over N = 2n synthetic
                         activation rows; along the channel axis X is an AR(1)
                         process (neighbouring channels correlated with rho) and
                         each channel is scaled by exp(0.5 z), z ~ N(0, 1)
                         (a spread of channel magnitudes like real activations).
  * ``hessian_diag``  -- fp32 [n] diagonal of such a Hessian without forming it:
                         channel energies exp(z) (the squared lognormal channel
                         scales), sampling noise of N = 2n rows in the normal
                         approximation of chi2_N / N, plus 1 % of the mean.
  * ``spectral_hessian`` -- fp64 symmetric Q diag(eigs) Q^T with Q orthogonal
                         from the QR factorisation of a seeded Gaussian matrix;
                         used to place the smallest eigenvalue exactly (e.g.
                         indefinite matrices for the damping retries).
"""
from __future__ import annotations

import math

import torch

# seeds of the sign vectors su / sv for a matrix drawn with seed `s`
SU_SEED_OFFSET = 1
SV_SEED_OFFSET = 2

DECODER_LAYER_PROJECTIONS = (
    # name, rows, cols  (rows = output features, cols = input features)
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 12288, 4096),
    ("up", 12288, 4096),
    ("down", 4096, 12288),
)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def iid_f32(rows: int, cols: int, seed: int = 0) -> torch.Tensor:
    return torch.randn(rows, cols, generator=_gen(seed), dtype=torch.float32)


def linear_bf16(rows: int, cols: int, seed: int = 0, std: float = 0.02,
                outlier_frac: float = 0.0, outlier_mult: float = 8.0) -> torch.Tensor:
    g = _gen(seed)
    w = torch.randn(rows, cols, generator=g, dtype=torch.float32) * std
    n_out = int(round(outlier_frac * rows * cols))
    if n_out > 0:
        idx = torch.randperm(rows * cols, generator=g)[:n_out]
        flat = w.view(-1)
        flat[idx] = flat[idx] * outlier_mult
    return w.to(torch.bfloat16)


def student_t_bf16(rows: int, cols: int, seed: int = 0, nu: int = 5,
                   std: float = 0.015) -> torch.Tensor:
    g = _gen(seed)
    z = torch.randn(rows, cols, generator=g, dtype=torch.float64)
    chi2 = torch.zeros(rows, cols, dtype=torch.float64)
    for _ in range(nu):
        chi2 += torch.randn(rows, cols, generator=g, dtype=torch.float64) ** 2
    t = z / torch.sqrt(chi2 / nu)
    t_std = math.sqrt(nu / (nu - 2.0))
    return (t * (std / t_std)).to(torch.float32).to(torch.bfloat16)


def signs(n: int, seed: int) -> torch.Tensor:
    b = torch.randint(0, 2, (n,), generator=_gen(seed), dtype=torch.int64)
    return (b * 2 - 1).to(torch.float32)


def sign_pair(rows: int, cols: int, seed: int):
    """(su[rows], sv[cols]) for a matrix drawn with seed `seed`."""
    return (signs(rows, seed + SU_SEED_OFFSET), signs(cols, seed + SV_SEED_OFFSET))


def workload(name: str):
    """Named workloads: returns a list of (label, W, su, sv, K) tuples.

    rot128_iid_k2   : one 128x128 fp32 N(0,1) matrix, already rotated (su, sv None), K=2.
    linear4096_k2   : 4096x4096 bf16 N(0, 0.02^2) with 0.1% outliers x8, K=2.
    mlp12288_t5_k4  : 12288x4096 bf16 Student-t(5) with std 0.015, K=4.
    layer4096_k3    : the 7 projections of one decoder layer, bf16 N(0, 0.02^2),
                      projection i drawn with seed i, K=3.
    gss4096_k2      : 4096x4096 bf16 N(0, 0.02^2), K=2 (golden-section search).
    """
    if name == "rot128_iid_k2":
        return [("rot128", iid_f32(128, 128, 0), None, None, 2)]
    if name == "linear4096_k2":
        W = linear_bf16(4096, 4096, 0, 0.02, outlier_frac=0.001, outlier_mult=8.0)
        return [("linear4096", W, *sign_pair(4096, 4096, 0), 2)]
    if name == "mlp12288_t5_k4":
        W = student_t_bf16(12288, 4096, 0, 5, 0.015)
        return [("mlp12288", W, *sign_pair(12288, 4096, 0), 4)]
    if name == "layer4096_k3":
        out = []
        for i, (lab, r, c) in enumerate(DECODER_LAYER_PROJECTIONS):
            W = linear_bf16(r, c, i, 0.02)
            su, sv = sign_pair(r, c, 100 + 2 * i)
            out.append((lab, W, su, sv, 3))
        return out
    if name == "gss4096_k2":
        W = linear_bf16(4096, 4096, 0, 0.02)
        return [("gss4096", W, *sign_pair(4096, 4096, 0), 2)]
    raise KeyError(name)


def spd_hessian(n: int, seed: int = 0, rho: float = 0.9, n_samples: int | None = None,
                damp: float = 0.01) -> torch.Tensor:
    g = _gen(seed)
    N = n_samples or 2 * n
    z = torch.randn(N, n, generator=g, dtype=torch.float64)
    x = torch.empty_like(z)
    x[:, 0] = z[:, 0]
    c = math.sqrt(1.0 - rho * rho)
    for k in range(1, n):
        x[:, k] = rho * x[:, k - 1] + c * z[:, k]
    x *= torch.exp(0.5 * torch.randn(n, generator=g, dtype=torch.float64))
    H = x.T @ x / N
    H = 0.5 * (H + H.T)
    H += damp * torch.diagonal(H).mean() * torch.eye(n, dtype=torch.float64)
    return H


def spectral_hessian(n: int, eigs, seed: int = 0) -> torch.Tensor:
    g = _gen(seed)
    q, r = torch.linalg.qr(torch.randn(n, n, generator=g, dtype=torch.float64))
    q = q * torch.sign(torch.diagonal(r))
    lam = torch.as_tensor(eigs, dtype=torch.float64)
    H = (q * lam) @ q.T
    return 0.5 * (H + H.T)


def hessian_diag(n: int, seed: int = 0, damp: float = 0.01) -> torch.Tensor:
    g = _gen(seed)
    energy = torch.exp(torch.randn(n, generator=g, dtype=torch.float64))
    noise = 1.0 + math.sqrt(2.0 / (2 * n)) * torch.randn(n, generator=g, dtype=torch.float64)
    h = energy * noise.clamp_min(0.0)
    h += damp * h.mean()
    return h.to(torch.float32)
