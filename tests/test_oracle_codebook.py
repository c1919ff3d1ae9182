"""Pins for the oracle's Lloyd-Max codebook (no GPU)."""

import math
import os

import numpy as np
import pytest
from scipy import integrate

from oracle import codebook

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _max_table():
    rows = {}
    with open(os.path.join(GOLDEN, "max1960_gaussian_quantizer.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = line.split()
            rows[int(v[0])] = (float(v[1]), [float(x) for x in v[2:]])
    return rows


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_one_bit_closed_form(d):
    c, b, mse, _ = codebook.lloyd_max(d, 1)
    # E|X| = Γ(d/2) / (√π Γ((d+1)/2)), evaluated in 30-digit arithmetic
    import mpmath as mp

    mp.mp.dps = 30
    want = float(mp.gamma(mp.mpf(d) / 2) / (mp.sqrt(mp.pi) * mp.gamma(mp.mpf(d + 1) / 2)))
    assert np.allclose(c, [-want, want], rtol=2e-15, atol=0)
    assert b.tolist() == [0.0]
    assert abs(mse - (1.0 / d - want * want)) < 1e-15


@pytest.mark.parametrize("d", [8, 128, 1024])
@pytest.mark.parametrize("w", [1, 2, 3])
def test_symmetry_and_midpoints(d, w):
    c, b, _, _ = codebook.lloyd_max(d, w)
    L = 1 << w
    assert len(c) == L and len(b) == L - 1
    assert np.array_equal(c, -c[::-1])
    assert np.all(np.diff(c) > 0)
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-16)


@pytest.mark.parametrize("d", [8, 128, 1024])
@pytest.mark.parametrize("w", [1, 2, 3])
def test_centroids_are_conditional_means_by_quadrature(d, w):
    """Independent adaptive quadrature of f_d reproduces every centroid and the MSE."""
    c, b, mse, _ = codebook.lloyd_max(d, w)
    edges = np.concatenate([[-1.0], b, [1.0]])
    k = codebook.density_const(d)
    a = (d - 3) / 2.0
    sd = 1.0 / math.sqrt(d)
    for i in range(len(c)):
        lo, hi = max(edges[i], -40 * sd), min(edges[i + 1], 40 * sd)
        m0 = integrate.quad(lambda x: k * (1 - x * x) ** a, lo, hi, epsabs=0, epsrel=1e-13, limit=500)[0]
        m1 = integrate.quad(lambda x: x * k * (1 - x * x) ** a, lo, hi, epsabs=0, epsrel=1e-13, limit=500)[0]
        assert abs(m1 / m0 - c[i]) < 1e-12 * sd * 10
    # MSE = 1/d - Σ p c² cancels down from E[X²] = 1/d: compare at 1e-12 of that scale
    assert abs(codebook.codebook_mse_numeric(c, b, d) - mse) < 1e-12 / d


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_mse_decreases_and_meets_printed_bounds(d):
    """4^-w ≤ d·MSE ≤ (√3·π/2)·4^-w (lower bound for any quantizer, upper bound for TurboQuant)."""
    prev = None
    for w in (1, 2, 3):
        _, _, mse, _ = codebook.lloyd_max(d, w)
        dm = d * mse
        assert 4.0 ** -w <= dm <= math.sqrt(3) * math.pi / 2 * 4.0 ** -w
        if prev is not None:
            assert dm < prev
        prev = dm


def test_one_bit_ratio_to_lower_bound_is_about_1_45():
    _, _, mse, _ = codebook.lloyd_max(1024, 1)
    assert abs(1024 * mse * 4.0 - 1.45) < 0.01


def test_large_d_tends_to_max_gaussian_quantizer():
    d = 100000
    table = _max_table()
    for w in (1, 2, 3):
        c, _, mse, _ = codebook.lloyd_max(d, w)
        want_mse, want_levels = table[1 << w]
        assert abs(d * mse - want_mse) < 2e-4
        got = math.sqrt(d) * c[len(c) // 2:]
        assert np.allclose(got, want_levels, rtol=0, atol=2e-3)


def test_lloyd_max_is_a_local_minimum():
    """Moving any centroid (with boundaries re-set to midpoints) raises the MSE by quadrature."""
    d, w = 128, 2
    c, b, mse, _ = codebook.lloyd_max(d, w)
    base = codebook.codebook_mse_numeric(c, b, d)
    for i in range(len(c)):
        for eps in (-1e-3, 1e-3):
            cc = c.copy()
            cc[i] += eps / math.sqrt(d)
            cc.sort()
            bb = 0.5 * (cc[:-1] + cc[1:])
            assert codebook.codebook_mse_numeric(cc, bb, d) > base


@pytest.mark.parametrize("d,w", [(128, 2), (128, 3), (1024, 3)])
def test_lloyd_conditions_hold_in_30_digit_arithmetic(d, w):
    """Centroid = conditional mean of its midpoint cell, checked by mpmath quadrature."""
    import mpmath as mp

    mp.mp.dps = 30
    c, _, _, _ = codebook.lloyd_max(d, w)
    half = len(c) // 2
    pos = [mp.mpf(float(v)) for v in c[half:]]
    edges = [mp.mpf(0)] + [(pos[k] + pos[k + 1]) / 2 for k in range(half - 1)] + [mp.mpf(1)]
    a = mp.mpf(d - 3) / 2
    for k in range(half):
        lo, hi = edges[k], edges[k + 1]
        m0 = mp.quad(lambda x: (1 - x * x) ** a, [lo, hi])
        m1 = mp.quad(lambda x: x * (1 - x * x) ** a, [lo, hi])
        assert abs(float(m1 / m0 - pos[k])) < 1e-12 * float(pos[-1])
