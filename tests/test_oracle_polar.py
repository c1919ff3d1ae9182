"""Pins for the oracle's PolarQuant stage (no GPU).

"TurboQuant 与 AI 效率革命" §二: recursive polar transform, angle density
Γ(k)/(2^(k-2)Γ(k/2)²)·sin^(k-1)(2ψ) with mean π/4; "TurboQuant压缩效果":
4 bits at the first level, 2 at later ones.
"""

import math

import numpy as np
import pytest
from scipy import integrate, stats

from oracle import polar, qjl, rotation


@pytest.mark.parametrize("k", [2, 4, 8, 64, 512])
def test_angle_density_integrates_to_one_with_mean_pi_over_4(k):
    tot, _ = integrate.quad(lambda p: polar.angle_density(p, k), 0, np.pi / 2, epsabs=1e-14, limit=400,
                            points=[np.pi / 4])
    mean, _ = integrate.quad(lambda p: p * polar.angle_density(p, k), 0, np.pi / 2, epsabs=1e-14, limit=400,
                             points=[np.pi / 4])
    assert abs(tot - 1.0) < 1e-10
    assert abs(mean - np.pi / 4) < 1e-10


@pytest.mark.parametrize("k", [2, 3, 8, 64])
def test_density_matches_the_incomplete_beta_cdf(k):
    """Two routes to P(ψ ≤ t): quadrature of the page's density, and the Beta(k/2, k/2) law of sin² ψ."""
    for t in np.linspace(0.05, np.pi / 2 - 0.05, 9):
        num, _ = integrate.quad(lambda p: polar.angle_density(p, k), 0, t, epsabs=1e-14, limit=400)
        assert abs(num - float(polar.angle_cdf(t, k))) < 1e-10


def test_angles_of_gaussian_vectors_follow_the_level_laws():
    """KS tests: level-1 angles uniform on [0, 2π), level-ℓ angles with CDF I_{sin²t}(k/2, k/2), k = 2^(ℓ-1)."""
    rng = np.random.default_rng(0)
    U = rng.standard_normal((4000, 128))
    radius, angles = polar.forward(U)
    assert np.allclose(radius, np.linalg.norm(U, axis=1), rtol=1e-13)
    a1 = angles[0].ravel()
    assert stats.kstest(a1, stats.uniform(loc=0, scale=2 * np.pi).cdf).pvalue > 1e-3
    for lev in range(2, 8):
        k = 1 << (lev - 1)
        a = angles[lev - 1].ravel()[:20000]
        assert stats.kstest(a, lambda t: polar.angle_cdf(t, k)).pvalue > 1e-3, lev


@pytest.mark.parametrize("d", [2, 8, 128])
def test_transform_round_trip_is_exact(d):
    rng = np.random.default_rng(d)
    U = rng.standard_normal((50, d))
    radius, angles = polar.forward(U)
    assert len(angles) == polar.levels(d) and sum(a.shape[1] for a in angles) == d - 1
    assert np.allclose(polar.inverse(radius, angles), U, rtol=1e-12, atol=1e-12)
    if d == 2:  # plain polar coordinates
        assert np.allclose(angles[0][:, 0], np.mod(np.arctan2(U[:, 1], U[:, 0]), 2 * np.pi))


@pytest.mark.parametrize("k", [2, 8, 64])
def test_lloyd_max_angle_codebook_meets_both_conditions(k):
    """Boundaries at midpoints; every centroid the conditional mean of its cell
    (independent quadrature of the density); symmetric about π/4."""
    c, b, mse = polar.lloyd_max_angle(k, 2)
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    edges = np.concatenate([[0.0], b, [np.pi / 2]])
    for j in range(len(c)):
        m0, _ = integrate.quad(lambda p: polar.angle_density(p, k), edges[j], edges[j + 1], epsabs=1e-15, limit=400)
        m1, _ = integrate.quad(lambda p: p * polar.angle_density(p, k), edges[j], edges[j + 1], epsabs=1e-15,
                               limit=400)
        assert abs(m1 / m0 - c[j]) < 1e-9
    assert np.allclose(c + c[::-1], np.pi / 2, atol=1e-9)
    assert mse < (np.pi / 2) ** 2 / 12 / 16  # far below a uniform 2-bit grid on [0, π/2]


def test_uniform_level_one_quantizer_distortion():
    """Equal cells of width Δ with midpoint centroids: MSE = Δ²/12 for a uniform angle."""
    c, b = polar.uniform_codebook(4)
    rng = np.random.default_rng(1)
    a = rng.uniform(0, 2 * np.pi, 400000)
    q = c[np.searchsorted(b, a, side="left")]
    delta = 2 * np.pi / 16
    assert abs(np.mean((a - q) ** 2) / (delta ** 2 / 12) - 1) < 0.01


def test_vectors_built_from_centroids_requantize_exactly():
    """x = Πᵀ inverse(R, centroids): every angle is its own centroid, so the indices
    come back, x̃ = x and the residual is zero (all signs +1)."""
    d = 16
    cb = polar.make_codebooks(d)
    Pi = rotation.make_rotation(d, 3)
    S = qjl.make_qjl(d, d, 4)
    rng = np.random.default_rng(2)
    N = 40
    idx = [rng.integers(0, len(c), size=(N, d >> lev)) for lev, (c, _) in enumerate(cb.books, start=1)]
    R = rng.uniform(0.5, 3.0, N)
    X = polar.reconstruct_stage1(idx, R, Pi, cb)
    q = polar.quantize_polar(X, Pi, S, cb)
    for got, want in zip(q.idx, idx):
        assert np.array_equal(got, want)
    assert np.allclose(polar.reconstruct(q, Pi, S, cb, qjl_stage=False), X, rtol=1e-6, atol=1e-6)
    assert np.all(q.rnorm < 1e-5 * R)


def test_bit_accounting():
    assert polar.bits_per_vector(128) == 64 * 4 + 63 * 2
    assert abs(polar.bits_per_vector(128) / 128 - 3.0) < 0.03
    assert polar.bits_per_vector(1024) == 512 * 4 + 511 * 2


def test_polar_plus_qjl_score_is_unbiased_over_qjl_draws():
    """The polar stage followed by QJL on its residual estimates ⟨q, x⟩ without
    bias: mean over 10^4 independent S within 3 standard errors."""
    d = 16
    cb = polar.make_codebooks(d)
    Pi = rotation.make_rotation(d, 7)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, d))
    qv = rng.standard_normal(d)
    est = np.empty(10000)
    for i in range(len(est)):
        S = rng.standard_normal((d, d))
        q = polar.quantize_polar(x, Pi, S, cb)
        est[i] = float(polar.reconstruct(q, Pi, S, cb)[0] @ qv)
    se = est.std(ddof=1) / math.sqrt(len(est))
    assert abs(est.mean() - float(x[0] @ qv)) < 3 * se


def test_index_packing_hand_pattern_and_round_trip():
    """d = 8, b1 = 4, b = 2: level-1 codes 1, 2, 3, 4 -> word 0 = 0x4321; level 2
    codes 3, 0 and level 3 code 2 -> word 1 = 3 | 0 << 2 | 2 << 4."""
    idx = [np.array([[1, 2, 3, 4]]), np.array([[3, 0]]), np.array([[2]])]
    w = polar.pack_indices(idx, 8)
    assert w.shape == (1, polar.index_words(8)) == (1, 2)
    assert int(w[0, 0]) == 0x4321 and int(w[0, 1]) == 3 | (2 << 4)
    rng = np.random.default_rng(5)
    for d in (4, 16, 128, 256):
        lv = [rng.integers(0, 16, size=(7, d // 2))] + [rng.integers(0, 4, size=(7, d >> l))
                                                         for l in range(2, polar.levels(d) + 1)]
        back = polar.unpack_indices(polar.pack_indices(lv, d), d)
        assert all(np.array_equal(a, b) for a, b in zip(lv, back))
    assert polar.index_words(128) == 8 + 4
