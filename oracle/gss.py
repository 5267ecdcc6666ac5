"""Golden-section scale search and one full evaluation (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the page "alpha2beta/JEV-9B-EXL3-K2", section 2 ("Quantization &
Bitrate Breakdown"): the scale of each quantized projection is chosen by golden
section search.  The page gives no bracket or iteration count; the search here
takes a bracket [lo, hi] and a total number of function evaluations.  Python
floats are IEEE binary64, so every step below is one binary64 operation.
"""
from __future__ import annotations

import math

import numpy as np


def golden_section_search(f, lo: float, hi: float, n_eval: int, return_bracket: bool = False):
    """Minimise f over [lo, hi] with exactly ``n_eval`` (>= 2) evaluations.

    phi = (sqrt(5) - 1) / 2.  Start with x1 = b - phi (b - a), x2 = a + phi (b - a)
    and evaluate both.  Then repeat: if f(x1) <= f(x2) the minimum lies in
    [a, x2]: b <- x2, x2 <- x1, x1 <- b - phi (b - a), evaluate x1; otherwise it
    lies in [x1, b]: a <- x1, x1 <- x2, x2 <- a + phi (b - a), evaluate x2.
    Returns (best_x, best_f, history) where best is the evaluated point with the
    least f, the smaller x on ties, and history lists (x, f) in evaluation order;
    with ``return_bracket`` also the final bracket (a, b).
    """
    if n_eval < 2:
        raise ValueError("golden-section search needs at least two evaluations")
    phi = (math.sqrt(5.0) - 1.0) / 2.0
    a, b = float(lo), float(hi)
    x1 = b - phi * (b - a)
    x2 = a + phi * (b - a)
    f1 = f(x1)
    f2 = f(x2)
    hist = [(x1, f1), (x2, f2)]
    n = 2
    while n < n_eval:
        if f1 <= f2:
            b = x2
            x2, f2 = x1, f1
            x1 = b - phi * (b - a)
            f1 = f(x1)
            hist.append((x1, f1))
        else:
            a = x1
            x1, f1 = x2, f2
            x2 = a + phi * (b - a)
            f2 = f(x2)
            hist.append((x2, f2))
        n += 1
    best_x, best_f = hist[0]
    for x, fx in hist[1:]:
        if fx < best_f or (fx == best_f and x < best_x):
            best_x, best_f = x, fx
    if return_bracket:
        return best_x, best_f, hist, (a, b)
    return best_x, best_f, hist


def evaluate_matrix(W, su, sv, K: int, g: float, threads: int | None = None):
    """One full evaluation at relative scale g: rotate, scale, encode, decode,
    inverse-rotate, MSE (quantizer README items 7, 1, 5, 10 in that order).

    W: fp32 [rows, cols] (a bf16 weight widened exactly).  Returns a dict with
    R, sigma, scale, inv_scale, states, costs, codes, Yhat, What, mse.
    """
    from . import (rotate_forward, rotate_inverse, rms, scale_for, encode_matrix,
                   codes_from_states, decode_matrix, mse)
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    R = rotate_forward(W, su, sv)
    sigma = rms(R)
    s, inv = scale_for(g, sigma)
    states, costs = encode_matrix(R, K, inv, threads=threads)
    codes = codes_from_states(states, rows, cols, K)
    Yhat = decode_matrix(codes, rows, cols, K, s)
    What = rotate_inverse(Yhat, su, sv)
    return dict(R=R, sigma=sigma, scale=s, inv_scale=inv, states=states, costs=costs,
                codes=codes, Yhat=Yhat, What=What, mse=mse(W, What))
