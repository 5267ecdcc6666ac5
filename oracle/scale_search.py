"""Grid-and-parabola global-scale search on a tile sample (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the page "EXL3 Intel Arc Quantizer", Core Implemented Architecture
item 8: the global scale is searched on a wrapped-diagonal sample of tiles plus
the highest- and lowest-RMS tiles, first on a coarse grid 0.1..1.9 over a
strided subsample, then on a fine grid within 0.075 of the coarse minimum over
the full sample, then refined by a parabola with a 0.01 floor.  The page gives
no more than that; the readings below fill in the rest, each a choice made
where the page is silent:

  * tiles are the 16x16 tiles of the rotated matrix R, TR x TC of them;
  * wrapped diagonal: tile (i mod TR, i mod TC) for i = 0 .. max(TR, TC) - 1;
    then the tile with the highest RMS and the one with the lowest RMS (per-tile
    fp64 sums of r^2, ties to the lower tile index), each appended only if it is
    not already in the sample;
  * the objective of a tile subset at relative scale g is the rotated-domain
    MSE: s = fl32(g * sigma_R), codes from y = fl(r * fl32(1/s)),
    err = sum over tiles and elements of (r - fl(v * s))^2 in fp64, each tile
    summed in row-major order, the tile sums added as a pairwise tree in sample
    order, divided by 256 * (number of tiles);
  * coarse grid g = k / 10, k = 1..19, on every second sample tile (indices
    0, 2, 4, ... of the sample);
  * fine grid g_c + 0.025 k, k = -3..3, on the full sample (g_c = coarse
    minimum, smaller g on ties; likewise below);
  * parabola through the fine minimum and its two grid neighbours (when the
    minimum is interior): the vertex of the interpolating parabola, floored at
    0.01; it is evaluated on the full sample and kept only if strictly better
    than the fine minimum.
"""
from __future__ import annotations

import numpy as np

COARSE = [k / 10.0 for k in range(1, 20)]
FINE_STEP = 0.025
FINE_K = range(-3, 4)
FLOOR = 0.01


def sample_tiles(tile_sums, TR: int, TC: int):
    """Wrapped diagonal, then the highest- and lowest-RMS tiles if new."""
    n = max(TR, TC)
    s = [(i % TR) * TC + (i % TC) for i in range(n)]
    ts = np.asarray(tile_sums, dtype=np.float64)
    hi = int(np.flatnonzero(ts == ts.max())[0])
    lo = int(np.flatnonzero(ts == ts.min())[0])
    for t in (hi, lo):
        if t not in s:
            s.append(t)
    return s


def parabola_vertex(a, fa, b, fb, c, fc):
    """Vertex of the parabola through (a, fa), (b, fb), (c, fc) (binary64);
    None when the three points are collinear."""
    p = (b - a) * (fb - fc)
    q = (b - c) * (fb - fa)
    den = p - q
    if den == 0.0:
        return None
    return b - 0.5 * ((b - a) * p - (b - c) * q) / den


def subset_mse(R, tiles, K: int, g: float, sigma: float):
    """Rotated-domain MSE of the listed tiles at relative scale g."""
    import oracle
    s, inv = oracle.scale_for(g, sigma)
    rows, cols = R.shape
    TC = cols // 16
    Y = np.empty((len(tiles), 256), dtype=np.float32)
    for j, t in enumerate(tiles):
        tr, tc = divmod(t, TC)
        Y[j] = R[tr * 16:(tr + 1) * 16, tc * 16:(tc + 1) * 16].reshape(-1)
    # encode each sampled tile as a 16 x 16 block of a [16, 16 * n] matrix
    M = np.concatenate([Y[j].reshape(16, 16) for j in range(len(tiles))], axis=1)
    states, _ = oracle.encode_matrix(M, K, inv)
    sums = np.empty(len(tiles), dtype=np.float64)
    for j in range(len(tiles)):
        yhat = oracle.decode_values(states[j], s)
        acc = 0.0
        for i in range(256):
            d = float(Y[j, i]) - float(yhat[i])
            acc = acc + d * d
        sums[j] = acc
    return oracle.tree_sum(sums) / (256.0 * len(tiles))


def grid_scale_search(R, K: int):
    """Returns dict(g, sigma, sample, coarse, fine, refined) with (g, mse) lists."""
    import oracle
    R = np.ascontiguousarray(R, dtype=np.float32)
    rows, cols = R.shape
    TR, TC = rows // 16, cols // 16
    ts = oracle.tile_sumsq(R)
    sigma = oracle.rms(R)
    S = sample_tiles(ts, TR, TC)
    Sc = S[0::2]
    coarse = [(g, subset_mse(R, Sc, K, g, sigma)) for g in COARSE]
    gc, fc = coarse[0]
    for g, f in coarse[1:]:
        if f < fc:
            gc, fc = g, f
    fine_g = [gc + FINE_STEP * k for k in FINE_K]
    fine = [(g, subset_mse(R, S, K, g, sigma)) for g in fine_g]
    ib = 0
    for i in range(1, len(fine)):
        if fine[i][1] < fine[ib][1]:
            ib = i
    gf, ff = fine[ib]
    refined = None
    g_final = gf
    if 0 < ib < len(fine) - 1:
        v = parabola_vertex(fine[ib - 1][0], fine[ib - 1][1], gf, ff, fine[ib + 1][0],
                            fine[ib + 1][1])
        if v is not None:
            v = max(v, FLOOR)
            fv = subset_mse(R, S, K, v, sigma)
            refined = (v, fv)
            if fv < ff:
                g_final = v
    return dict(g=g_final, sigma=sigma, sample=S, coarse=coarse, fine=fine, refined=refined)
