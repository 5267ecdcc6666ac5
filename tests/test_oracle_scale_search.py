"""Pins for the oracle's grid-and-parabola scale search (not gpu).

Page "EXL3 Intel Arc Quantizer", Core Implemented Architecture item 8 and the
test list's gss entry ("MSE-below-g_scale=1", determinism, floor/basin of the
refinement).  The readings of the unstated details are in oracle/scale_search.py.
"""
import numpy as np
import pytest

import oracle
from oracle import scale_search as ss


@pytest.mark.parametrize("xstar,a,h", [(0.62, 0.5, 0.25), (1.37, 1.3, 0.025), (0.4, 0.35, 0.05)])
def test_parabola_vertex_of_exact_quadratics(xstar, a, h):
    f = lambda x: 3.0 * (x - xstar) ** 2 + 0.5
    v = ss.parabola_vertex(a, f(a), a + h, f(a + h), a + 2 * h, f(a + 2 * h))
    assert abs(v - xstar) < 1e-9
    assert ss.parabola_vertex(0.25, 1.0, 0.5, 2.0, 0.75, 3.0) is None  # collinear (exact in binary)


def test_wrapped_diagonal_covers_rows_and_columns_and_adds_extremes():
    TR, TC = 4, 6
    ts = np.arange(TR * TC, dtype=np.float64) + 1.0
    ts[7] = 100.0      # (1, 1): on the diagonal -> not duplicated
    ts[2] = 0.0        # (0, 2): off the diagonal -> appended
    S = ss.sample_tiles(ts, TR, TC)
    diag = S[:6]
    assert diag == [0, 7, 14, 21, 4, 11]
    assert {t // TC for t in diag} == set(range(TR)) and {t % TC for t in diag} == set(range(TC))
    assert S[6:] == [2]
    # ties go to the lower tile index
    ts2 = np.ones(TR * TC)
    ts2[[3, 9]] = 5.0
    assert ss.sample_tiles(ts2, TR, TC)[6] == 3


@pytest.fixture(scope="module")
def small_search():
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((128, 128)) * 0.02).astype(np.float32)
    su = rng.choice([-1.0, 1.0], 128).astype(np.float32)
    sv = rng.choice([-1.0, 1.0], 128).astype(np.float32)
    R = oracle.rotate_forward(W, su, sv)
    return R, ss.grid_scale_search(R, 2)


def test_search_structure_and_mse_below_unit_scale(small_search):
    R, res = small_search
    assert [g for g, _ in res["coarse"]] == [k / 10.0 for k in range(1, 20)]
    gc = min(res["coarse"], key=lambda p: (p[1], p[0]))[0]
    assert [g for g, _ in res["fine"]] == [gc + 0.025 * k for k in range(-3, 4)]
    f_final = ss.subset_mse(R, res["sample"], 2, res["g"], res["sigma"])
    f_one = ss.subset_mse(R, res["sample"], 2, 1.0, res["sigma"])
    assert f_final <= f_one
    assert res["g"] >= 0.01
    fine_best = min(f for _, f in res["fine"])
    if res["refined"] is not None and res["refined"][1] < fine_best:
        assert res["g"] == res["refined"][0]
    else:
        assert res["g"] in [g for g, _ in res["fine"]]


def test_search_is_deterministic(small_search):
    R, res = small_search
    again = ss.grid_scale_search(R, 2)
    assert again["coarse"] == res["coarse"] and again["fine"] == res["fine"] and again["g"] == res["g"]
