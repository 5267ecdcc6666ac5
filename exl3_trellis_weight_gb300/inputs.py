"""Seeded synthetic inputs for tests and benchmarks.

This module draws random numbers only; it holds none of the encoder's
arithmetic.  Both the CUDA path and the CPU oracle are fed the very same
tensors produced here, so a comparison never depends on how either side draws.
The weight workloads and sign vectors come from a counter-based SplitMix64
stream through integer and correctly rounded binary64 operations only, so
every host (x86 or Arm) draws the same bytes and stored expected values
written on one host hold on another; the Hessian stand-ins, used only where
both sides are fed on the same host, are drawn with a seeded
``torch.Generator``.

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

import numpy as np
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


# --------------------------------------------------------------------------
# counter-based stream for the weight workloads
# --------------------------------------------------------------------------
# The weight matrices and sign vectors must be the same bytes on every host
# (an x86 container writes stored expected values; an Arm host re-draws the
# inputs and checks them), so they are drawn with integer arithmetic and
# correctly rounded IEEE binary64 operations only (+, -, *, /, sqrt, frexp);
# no library transcendental, whose last bits differ between platforms.
#
# Stream: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
# number generators", OOPSLA 2014; the reference code by S. Vigna): output i
# (i = 0, 1, ...) of the stream with seed s is mix(s + (i + 1) * gamma mod 2^64),
#   mix(z): z = (z ^ z >> 30) * 0xBF58476D1CE4E5B9; z = (z ^ z >> 27) *
#           0x94D049BB133111EB; return z ^ z >> 31.
# Uniform (0, 1): (2 * (u >> 12) + 1) * 2^-53, an odd multiple of 2^-53.
# Normal: Marsaglia's polar method (Marsaglia and Bray 1964) on consecutive
# pairs, with ln evaluated as e ln2 + 2 atanh((m - 1)/(m + 1)) from frexp.
# Normals are drawn in blocks of a fixed number of pairs; a draw of n values
# consumes whole blocks (the accepted values of block 0, then block 1, ...,
# cut at n), so blocks can be computed on several threads without changing a
# single output.

_MASK64 = (1 << 64) - 1
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_LN2 = 0.6931471805599453
_SQRT_HALF = 0.7071067811865476
# 1 / (2k + 1), k = 0..8: the series atanh(z) / z = sum z^(2k) / (2k + 1),
# truncated where z^18 / 19 < 1e-28 for |z| < 0.1716
_ATANH_COEF = tuple(1.0 / (2 * k + 1) for k in range(9))
_PAIRS_PER_BLOCK = 1 << 19
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import os
        from concurrent.futures import ThreadPoolExecutor
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _mix64(z: np.ndarray) -> np.ndarray:
    z ^= z >> np.uint64(30)
    z *= _MIX1
    z ^= z >> np.uint64(27)
    z *= _MIX2
    z ^= z >> np.uint64(31)
    return z


def _ln(x: np.ndarray) -> np.ndarray:
    """Natural log of positive finite binary64 values, from basic operations only
    (relative error below 1e-15; what matters here is that it is the same bits
    on every IEEE host)."""
    m, e = np.frexp(x)                       # x = m 2^e, m in [0.5, 1)
    lo = m < _SQRT_HALF
    m = np.where(lo, m * 2.0, m)             # m in [sqrt(1/2), sqrt(2))
    e = np.where(lo, e - 1, e).astype(np.float64)
    z = (m - 1.0) / (m + 1.0)                # |z| < 0.1716
    z2 = z * z
    p = np.full_like(z, _ATANH_COEF[-1])
    for c in _ATANH_COEF[-2::-1]:
        p *= z2
        p += c
    z *= 2.0
    p *= z
    e *= _LN2
    e += p
    return e


def _u64_at(seed: np.uint64, first: int, n: int) -> np.ndarray:
    """Stream outputs first .. first + n - 1 (0-based)."""
    i = np.arange(first + 1, first + 1 + n, dtype=np.uint64)
    i *= _GAMMA
    i += seed
    return _mix64(i)


def _polar_block(seed: np.uint64, first: int) -> np.ndarray:
    u = (_u64_at(seed, first, 2 * _PAIRS_PER_BLOCK) >> np.uint64(12)).astype(np.float64)
    u *= 2.0
    u += 1.0
    u *= 2.0 ** -53                          # uniform (0, 1), exact
    u *= 2.0
    u -= 1.0                                 # uniform (-1, 1), exact
    a, b = u[0::2], u[1::2]
    s = a * a + b * b
    ok = s < 1.0
    a, b, s = a[ok], b[ok], s[ok]
    f = np.sqrt((_ln(s) * -2.0) / s)
    z = np.empty(2 * s.size, dtype=np.float64)
    np.multiply(a, f, out=z[0::2])
    np.multiply(b, f, out=z[1::2])
    return z


class Stream:
    """SplitMix64 stream with seed ``seed`` (see above); draws advance a counter."""

    def __init__(self, seed: int):
        self.seed = np.uint64(int(seed) & _MASK64)
        self.pos = 0

    def u64(self, n: int) -> np.ndarray:
        out = _u64_at(self.seed, self.pos, n)
        self.pos += n
        return out

    def uniform(self, n: int) -> np.ndarray:
        """n values (2 (u >> 12) + 1) 2^-53 in (0, 1), binary64."""
        k = (self.u64(n) >> np.uint64(12)).astype(np.float64)
        return (k * 2.0 + 1.0) * (2.0 ** -53)

    def normal(self, n: int) -> np.ndarray:
        """n standard normals (binary64) by the polar method: for each pair
        (a, b) = 2U - 1 with 0 < s = a^2 + b^2 < 1, emit a f, b f where
        f = sqrt(-2 ln(s) / s); rejected pairs emit nothing."""
        out = np.empty(n, dtype=np.float64)
        filled, blk = 0, 0
        per_block = 2 * _PAIRS_PER_BLOCK
        while filled < n:
            # expected yield pi/4 per pair; ask for a few blocks more than that
            want = max(1, int((n - filled) / (per_block * 0.78)) + 1)
            firsts = [self.pos + (blk + j) * per_block for j in range(want)]
            for z in _pool().map(lambda f: _polar_block(self.seed, f), firsts):
                blk += 1
                take = min(n - filled, z.size)
                out[filled:filled + take] = z[:take]
                filled += take
                if filled == n:
                    break
        self.pos += blk * per_block
        return out

    def sample_without_replacement(self, population: int, k: int) -> np.ndarray:
        """k distinct indices of range(population): a partial Fisher-Yates shuffle,
        step i swapping position i with i + (u_i mod (population - i))."""
        r = self.u64(k)
        swapped: dict[int, int] = {}
        out = np.empty(k, dtype=np.int64)
        for i in range(k):
            j = i + int(r[i]) % (population - i)
            vi = swapped.get(i, i)
            out[i] = swapped.get(j, j)
            swapped[j] = vi
        return out


def _to_bf16(x64: np.ndarray, shape) -> torch.Tensor:
    """binary64 -> fp32 (round to nearest) -> bf16 (round to nearest even)."""
    f32 = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float64).astype(np.float32))
    return f32.reshape(shape).to(torch.bfloat16)


def iid_f32(rows: int, cols: int, seed: int = 0) -> torch.Tensor:
    z = Stream(seed).normal(rows * cols)
    return torch.from_numpy(z.astype(np.float32).reshape(rows, cols))


def linear_bf16(rows: int, cols: int, seed: int = 0, std: float = 0.02,
                outlier_frac: float = 0.0, outlier_mult: float = 8.0) -> torch.Tensor:
    st = Stream(seed)
    w = (st.normal(rows * cols) * float(std)).astype(np.float32)
    n_out = int(round(outlier_frac * rows * cols))
    if n_out > 0:
        idx = st.sample_without_replacement(rows * cols, n_out)
        w[idx] = w[idx] * np.float32(outlier_mult)
    return torch.from_numpy(w.reshape(rows, cols)).to(torch.bfloat16)


def student_t_bf16(rows: int, cols: int, seed: int = 0, nu: int = 5,
                   std: float = 0.015) -> torch.Tensor:
    """t = z / sqrt(chi2_nu / nu), chi2_nu = n_1^2 + ... + n_nu^2 summed in that
    order; z for every entry is drawn first, then n_1 for every entry, and so on."""
    st = Stream(seed)
    n = rows * cols
    z = st.normal(n)
    chi2 = np.zeros(n, dtype=np.float64)
    for _ in range(nu):
        x = st.normal(n)
        chi2 += x * x
    t = z / np.sqrt(chi2 / float(nu))
    t_std = math.sqrt(nu / (nu - 2.0))
    return _to_bf16(t * (std / t_std), (rows, cols))


def signs(n: int, seed: int) -> torch.Tensor:
    """n independent +-1 (fp32): the top bit of each stream output."""
    b = (Stream(seed).u64(n) >> np.uint64(63)).astype(np.float32)
    return torch.from_numpy(b * 2.0 - 1.0)


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
