"""Pins of the oracle's per-iteration coefficient schedule ("Polar Express" option)
to mathematics that does not go through it.

The schedule fits, at each iteration, the odd quintic closest to 1 in the max norm
on the current singular-value interval. These tests check, on grids and
perturbations the solver never sees, the properties that characterise that
polynomial:
- the error alternates four times at its maximum (Chebyshev equioscillation for a
  three-function basis);
- no nearby coefficients do better;
- the next interval is the image of this one;
- the limit on a point interval at 1 is the quintic flat to third order there.

Newton-Schulz with the schedule matches the SVD closed form with a different
polynomial at each step. A wrong sign, a transposed coefficient order or a lost
interval update fails one of them.
"""
import math

import numpy as np
import pytest

import oracle

EPS = 1e-7
LOWER = 1e-3


def _poly(co, x):
    a, b, c = co
    return a * x + b * x ** 3 + c * x ** 5


def _intervals(n, lower=LOWER):
    co, errs = oracle.polar_express_schedule(n, lower)
    spans, lo, hi = [], lower, 1.0
    for e in errs:
        spans.append((lo, hi))
        lo, hi = 1.0 - e, 1.0 + e
    return co, errs, spans


@pytest.mark.parametrize("k", range(6))
def test_error_equioscillates_at_its_maximum(k):
    co, errs, spans = _intervals(6)
    lo, hi = spans[k]
    x = np.linspace(lo, hi, 1_000_003)          # a grid unlike the solver's
    err = 1.0 - _poly(co[k], x)
    E = errs[k]
    assert abs(np.max(np.abs(err)) - E) <= 1e-8 * max(E, 1e-12) + 1e-15
    # four points of alternating sign at (nearly) the maximum, in order along x
    near = np.where(np.abs(err) >= E * (1 - 1e-6))[0]
    signs = np.sign(err[near])
    alternations = 1 + int(np.sum(signs[1:] != signs[:-1]))
    assert alternations >= 4


@pytest.mark.parametrize("k", range(5))
def test_no_nearby_quintic_does_better(k):
    co, errs, spans = _intervals(5)
    lo, hi = spans[k]
    x = np.linspace(lo, hi, 200_003)
    best = np.max(np.abs(1.0 - _poly(co[k], x)))
    rng = np.random.default_rng(k)
    base = np.array(co[k])
    for scale in (1e-3, 1e-5):
        for _ in range(100):
            trial = base * (1.0 + scale * rng.standard_normal(3))
            assert np.max(np.abs(1.0 - _poly(trial, x))) >= best * (1 - 1e-9)


def test_next_interval_is_the_image_of_this_one():
    co, errs, spans = _intervals(6)
    for k in range(5):
        lo, hi = spans[k]
        y = _poly(co[k], np.linspace(lo, hi, 500_001))
        assert abs(y.min() - (1 - errs[k])) <= 1e-7
        assert abs(y.max() - (1 + errs[k])) <= 1e-7
        assert spans[k + 1] == pytest.approx((1 - errs[k], 1 + errs[k]), abs=0)


def test_limit_is_the_quintic_flat_to_third_order_at_one():
    # p(1) = 1, p'(1) = 0, p''(1) = 0 for p = a x + b x^3 + c x^5
    M = np.array([[1.0, 1.0, 1.0], [1.0, 3.0, 5.0], [0.0, 6.0, 20.0]])
    flat = np.linalg.solve(M, [1.0, 0.0, 0.0])
    co, errs = oracle.polar_express_schedule(9, LOWER)
    assert np.allclose(co[-1], flat, rtol=0, atol=1e-6)
    assert errs[-1] < 1e-12


def test_errors_fall_and_fewer_iterations_match_the_fixed_quintic():
    # the aim the pages give: fewer iterations to the same polar accuracy.  The
    # fixed quintic's five steps leave max |1 - P(x)| on [1e-3, 1] at about 0.53
    x = np.linspace(LOWER, 1.0, 400_001)
    y = x.copy()
    for _ in range(5):
        y = _poly(oracle.DEFAULT_COEFFS, y)
    fixed5 = float(np.max(np.abs(1.0 - y)))
    co, errs = oracle.polar_express_schedule(5, LOWER)
    assert all(e1 < e0 for e0, e1 in zip(errs, errs[1:]))
    comp = x.copy()
    dev = []
    for k in range(5):
        comp = _poly(co[k], comp)
        dev.append(float(np.max(np.abs(1.0 - comp))))
    assert dev == pytest.approx(errs, rel=1e-9)
    # dev[k] follows k + 1 steps
    assert dev[3] < fixed5 * 1.05   # four steps: about the fixed quintic's five
    assert dev[4] < fixed5 / 4      # five steps: well inside them


@pytest.mark.parametrize("shape", [(7, 11), (16, 16), (30, 9)])
def test_schedule_matches_svd_closed_form(shape):
    V = np.random.default_rng(3).standard_normal(shape)
    co, _ = oracle.polar_express_schedule(5, LOWER)
    P, s, Qt = np.linalg.svd(V, full_matrices=False)
    x = s / (math.sqrt(float(np.sum(s ** 2))) + EPS)
    for t in co:
        x = _poly(t, x)
    want = (P * x) @ Qt
    got = oracle.newton_schulz(V, steps=5, coeffs=co, eps=EPS)
    assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)


def test_schedule_of_one_triple_is_the_fixed_iteration():
    V = np.random.default_rng(4).standard_normal((12, 20))
    fixed = oracle.newton_schulz(V, steps=4)
    listed = oracle.newton_schulz(V, steps=4, coeffs=[oracle.DEFAULT_COEFFS] * 4)
    assert np.array_equal(fixed, listed)


def test_short_schedule_repeats_its_last_triple():
    co = [(1.5, -0.5, 0.0), (1.875, -1.25, 0.375)]
    assert oracle.coefficient_schedule(co, 4) == [co[0], co[1], co[1], co[1]]
    V = np.random.default_rng(5).standard_normal((6, 9))
    a = oracle.newton_schulz(V, steps=4, coeffs=co)
    b = oracle.newton_schulz(V, steps=4, coeffs=[co[0], co[1], co[1], co[1]])
    assert np.array_equal(a, b)


def test_safety_widens_the_fitted_interval():
    co1, e1 = oracle.polar_express_schedule(3, LOWER, safety=1.0)
    co2, e2 = oracle.polar_express_schedule(3, LOWER, safety=1.05)
    # a wider interval cannot be fitted better
    assert e2[0] > e1[0]
    # and the safer polynomial keeps [l, 1.05] inside its error band
    x = np.linspace(LOWER, 1.05, 200_001)
    assert np.max(np.abs(1.0 - _poly(co2[0], x))) <= e2[0] * (1 + 1e-8)
