"""Pins of the oracle's phi functions (eq. (6) and (7) of "Continuous Softmax
Attention", section "Preliminaries") against things other than the oracle:
the values the page prints, the integral definitions evaluated by adaptive
quadrature, and the closed forms evaluated in 60-digit arithmetic."""
import math
import os

import mpmath
import pytest

import oracle

mpmath.mp.dps = 60

GRID = [0.0, 1e-12, -1e-12, 1e-8, -1e-8, 1e-3, -1e-3, 0.05, -0.05, 0.0999, -0.0999, 0.1, -0.1,
        0.3, -0.3, 0.5, -0.5, 1.0, -1.0, 1.0001, -1.0001, 3.0, -3.0, 10.0, -10.0, 40.0, -40.0,
        88.0, -88.0, 200.0, -200.0, 700.0, -700.0]


def _golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "phi_limits.txt")
    rows = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, x, val = line.split()
            rows[name] = (float(x), float(val))
    return rows


def test_limits_printed_on_the_page():
    g = _golden()
    assert oracle.phi1(g["phi1"][0]) == g["phi1"][1]
    assert oracle.phi2(g["phi2"][0]) == g["phi2"][1]


def _mp_phi1(x):
    x = mpmath.mpf(x)
    if x == 0:
        return mpmath.mpf(1)
    return mpmath.expm1(x) / x


def _mp_phi2(x):
    x = mpmath.mpf(x)
    if x == 0:
        return mpmath.mpf(1) / 2
    return (mpmath.expm1(x) - x) / (x * x)


@pytest.mark.parametrize("x", GRID)
def test_phi_against_high_precision(x):
    if abs(x) <= 700:
        assert oracle.phi1(x) == pytest.approx(float(_mp_phi1(x)), rel=2e-15, abs=0)
        assert oracle.phi2(x) == pytest.approx(float(_mp_phi2(x)), rel=2e-15, abs=0)
    assert oracle.log_phi1(x) == pytest.approx(float(mpmath.log(_mp_phi1(x))), rel=1e-14, abs=1e-15)
    assert oracle.log_phi2(x) == pytest.approx(float(mpmath.log(_mp_phi2(x))), rel=1e-14, abs=1e-15)


@pytest.mark.parametrize("x", [-30.0, -4.0, -0.7, -1e-4, 0.0, 2e-4, 0.6, 5.0, 25.0])
def test_phi_against_integral_definition(x):
    """eq. (6) defines phi1, phi2 as integrals over s in [0, 1]."""
    i1 = mpmath.quad(lambda s: mpmath.exp(s * x), [0, 1])
    i2 = mpmath.quad(lambda s: mpmath.exp(s * x) * (1 - s), [0, 1])
    assert oracle.phi1(x) == pytest.approx(float(i1), rel=1e-14)
    assert oracle.phi2(x) == pytest.approx(float(i2), rel=1e-14)


@pytest.mark.parametrize("x", [s * 10.0 ** e for e in range(-9, 3) for s in (1.0, -1.0, 3.7, -3.7)])
def test_identity_7(x):
    """eq. (7): phi1(x) - phi2(x) = e^x phi2(-x)."""
    lhs = oracle.phi1(x) - oracle.phi2(x)
    rhs = math.exp(x) * oracle.phi2(-x)
    assert lhs == pytest.approx(rhs, rel=1e-13)


@pytest.mark.parametrize("x", GRID + [1e4, -1e4, 1e6, -1e6])
def test_positivity_and_finite_logs(x):
    """End of "Preliminaries": phi1, phi2 > 0, so their logs are defined."""
    assert math.isfinite(oracle.log_phi2(x))
    assert math.isfinite(oracle.log_phi1(x))
    if abs(x) <= 700:
        assert oracle.phi2(x) > 0 and oracle.phi1(x) > 0


def test_series_branch_continuity():
    """The series (|x| < 0.1) and the closed form meet without a jump."""
    for x0 in (0.1, -0.1):
        lo = oracle.phi2(math.nextafter(x0, 0.0))
        hi = oracle.phi2(x0)
        assert hi == pytest.approx(lo, rel=1e-14)
