"""Output-channel regularisation of a weight before rotation (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the page "EXL3 Intel Arc Quantizer", Core Implemented Architecture
item 8 ("Weight Regularization & Global-Scale Search"): block_rms with a
32-slice accumulation order, the output-scale skew heuristic (the top 2 % of
sqrt(H_diag) against a 15 % cutoff), output-channel RMS normalisation, sign and
scale folded into sv, and the zero-channel floor 0.1 with sv = 0.  The page
names these parts only; the readings below fill in the rest, each a choice
made where the page is silent:

  * W [rows, cols] has the input channels down the rows (the Hessian's index)
    and the output channels across; H_diag [rows] is the Hessian's diagonal;
  * block_rms of output channel c: the rows cut into 32 consecutive slices of
    ceil(rows / 32), each slice's binary64 sum of squares in row order, the
    slice sums added in slice order (S_c); rms_c = fl32(sqrt(S_c / rows));
  * skew: d = sqrt(H_diag) in binary64 sorted descending, m = max(1, rows // 50)
    (2 %); skew = tree(first m) / tree(all), each a binary64 pairwise tree
    (neighbours (2i, 2i+1) per level, an odd last element moves up) over the
    sorted values, 0 when the total is 0; output scales are applied when
    skew < 0.15 (a flat input spectrum), otherwise every channel takes the
    global RMS fl32(sqrt(tree(S) / (rows * cols))) (S added as a pairwise tree);
  * a channel with S_c = 0 takes the floor scale 0.1 and sv = 0 (it decodes to
    zero whatever its codes); the weight is all zero ("zeros") when every S_c
    is 0;
  * W_out = fl32(W / scale_c) column by column; sv_out = sv * scale_c.
"""
from __future__ import annotations

import numpy as np

SLICES = 32
TOP_DIV = 50          # top 2 %
CUTOFF = 0.15
ZERO_FLOOR = 0.1


def block_sumsq_cols(W, slices: int = SLICES) -> np.ndarray:
    from oracle import _load, _p
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    out = np.empty(cols, dtype=np.float64)
    _load().ora_block_sumsq_cols(_p(W), rows, cols, int(slices), _p(out))
    return out


def skew(h) -> float:
    import oracle
    d = np.sqrt(np.asarray(h, dtype=np.float32).astype(np.float64))
    d = np.ascontiguousarray(np.sort(d)[::-1])
    m = max(1, d.size // TOP_DIV)
    total = oracle.tree_sum(d)
    return 0.0 if total == 0.0 else oracle.tree_sum(d[:m]) / total


def regularize(W, h, sv, apply_out: int = -1):
    """Returns dict(W_out, sv_out, skew, apply_out, zeros, rms)."""
    import oracle
    W = np.ascontiguousarray(W, dtype=np.float32)
    sv = np.asarray(sv, dtype=np.float32)
    rows, cols = W.shape
    S = block_sumsq_cols(W)
    sk = skew(h)
    app = (sk < CUTOFF) if apply_out < 0 else bool(apply_out)
    total = oracle.tree_sum(S)
    g_rms = np.float32(np.sqrt(total / float(rows * cols)))
    scale = np.empty(cols, dtype=np.float32)
    for c in range(cols):
        if S[c] == 0.0:
            scale[c] = np.float32(ZERO_FLOOR)
        elif app:
            scale[c] = np.float32(np.sqrt(S[c] / float(rows)))
        else:
            scale[c] = g_rms
    W_out = (W / scale[None, :]).astype(np.float32)        # fp32 division, one rounding
    sv_out = np.where(S == 0.0, np.float32(0.0), sv * scale).astype(np.float32)
    return dict(W_out=W_out, sv_out=sv_out, skew=sk, apply_out=app, zeros=bool(total == 0.0),
                rms=float(g_rms))
