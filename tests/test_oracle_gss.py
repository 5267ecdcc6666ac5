"""Pins for the oracle's golden-section search (not gpu).

Page "alpha2beta/JEV-9B-EXL3-K2", section 2: scale chosen by golden section
search.  For a unimodal f the minimiser stays inside the bracket, which shrinks
by phi = (sqrt 5 - 1)/2 per evaluation after the first two, so after n
evaluations the best evaluated point is within (hi - lo) * phi^(n-1) of it.
"""
import math

import numpy as np
import pytest

import oracle

PHI = (math.sqrt(5.0) - 1.0) / 2.0


@pytest.mark.parametrize("xstar", [0.5, 0.61, 0.9, 1.0, 1.37, 1.9, 2.0])
@pytest.mark.parametrize("n", [2, 3, 5, 12])
def test_quadratic_minimiser_within_textbook_bound(xstar, n):
    f = lambda x: (x - xstar) ** 2
    best, fb, hist = oracle.golden_section_search(f, 0.5, 2.0, n)
    assert len(hist) == n
    assert abs(best - xstar) <= 1.5 * PHI ** (n - 1) + 1e-12
    assert fb == min(h[1] for h in hist)


def test_first_points_and_shrink_ratio():
    seen = []
    f = lambda x: (seen.append(x), (x - 0.7) ** 2)[1]
    oracle.golden_section_search(f, 0.5, 2.0, 12)
    assert abs(seen[0] - (0.5 + (1 - PHI) * 1.5)) < 1e-15
    assert abs(seen[1] - (0.5 + PHI * 1.5)) < 1e-15
    # every later point is an interior golden point of the current bracket:
    # it lies strictly inside [0.5, 2.0] and differs from all earlier points
    assert all(0.5 < x < 2.0 for x in seen)
    assert len(set(seen)) == len(seen)


def test_tie_prefers_smaller_x_and_determinism():
    f = lambda x: 1.0
    a = oracle.golden_section_search(f, 0.5, 2.0, 12)
    b = oracle.golden_section_search(f, 0.5, 2.0, 12)
    assert a == b
    assert a[0] == min(h[0] for h in a[2])


def test_rejects_fewer_than_two_evaluations():
    with pytest.raises(ValueError):
        oracle.golden_section_search(lambda x: x, 0.5, 2.0, 1)


def test_unit_scale_inside_the_final_bracket_can_beat_the_best_point():
    """Golden-section search assumes a unimodal objective; the quantisation MSE
    as a function of the relative scale g is not unimodal at fine resolution, so
    'MSE(best g) <= MSE(g = 1) whenever g = 1 is inside the final bracket' is not
    a property of the search.  Pinned counterexample (K = 2, 128x128, seed 42, six
    evaluations): g = 1 lies inside the final bracket and codes with a lower MSE
    than every evaluated point.  The check 'MSE at the chosen scale <= MSE at
    unit scale' belongs to the page-1 grid search, where g = 1 is a grid point
    (tests/test_oracle_scale_search.py)."""
    from exl3_trellis_weight_gb300 import inputs
    W = inputs.linear_bf16(128, 128, seed=42, std=0.02)
    su, sv = inputs.sign_pair(128, 128, 42)
    Wf, sun, svn = W.float().numpy(), su.numpy(), sv.numpy()

    def f(g):
        return oracle.evaluate_matrix(Wf, sun, svn, 2, g)["mse"]

    best_g, best_f, hist, (a, b) = oracle.golden_section_search(f, 0.5, 2.0, 6, return_bracket=True)
    assert len(hist) == 6 and a < 1.0 < b
    assert best_f == min(y for _, y in hist)
    assert f(1.0) < best_f
