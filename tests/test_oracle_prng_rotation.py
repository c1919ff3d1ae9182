"""Pins for the oracle's generator and rotation (no GPU)."""

import os

import numpy as np
import pytest
from scipy import stats

from oracle import prng, rotation

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_ints(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(x) for x in f.read().split("\n") if x and not x.startswith("#")]


def test_splitmix64_published_sequence():
    want = _golden_ints("splitmix64_seed1234567.txt")
    got = [int(v) for v in prng.splitmix64(1234567, 5)]
    assert got == want


def test_splitmix64_offset_stream_is_counter_based():
    a = prng.splitmix64(99, 10)
    b = prng.splitmix64(99, 4, start=6)
    assert np.array_equal(a[6:], b)


def test_uniforms_open_interval_and_moments():
    u = prng.uniforms(7, 1 << 16)
    assert u.min() > 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3


def test_box_muller_normals_are_standard_normal():
    z = prng.normals(12345, 1 << 16)
    assert abs(z.mean()) < 4.0 / 256
    assert abs(z.var() - 1.0) < 0.03
    assert stats.kstest(z, "norm").pvalue > 1e-3
    # the two members of a pair are independent: uncorrelated, and z₁² + z₂² ~ Exp(mean 2)
    z1, z2 = z[0::2], z[1::2]
    assert abs(np.corrcoef(z1, z2)[0, 1]) < 4.0 / np.sqrt(len(z1))
    assert stats.kstest(z1 * z1 + z2 * z2, "expon", args=(0.0, 2.0)).pvalue > 1e-3
    # odd count is a prefix of the even fill
    assert np.array_equal(prng.normals(12345, 7), z[:7])


@pytest.mark.parametrize("d", [8, 32, 128, 1024])
def test_rotation_is_orthogonal_and_norm_preserving(d):
    P = rotation.make_rotation(d, 0x71550001)
    assert np.abs(P @ P.T - np.eye(d)).max() < 1e-13
    x = prng.normals(5, 3 * d).reshape(3, d)
    nx = np.linalg.norm(x, axis=1)
    nu = np.linalg.norm(x @ P.T, axis=1)
    assert np.max(np.abs(nu / nx - 1.0)) < 1e-12


@pytest.mark.parametrize("d", [8, 128])
def test_rotation_is_the_positive_diagonal_qr_factor(d):
    """Πᵀ G must be upper triangular with a positive diagonal (unique QR)."""
    seed = 0x1234 + d
    P = rotation.make_rotation(d, seed)
    G = prng.gaussian_matrix(seed, d, d)
    R = P.T @ G
    assert np.abs(np.tril(R, -1)).max() < 1e-10 * np.abs(R).max()
    assert np.all(np.diag(R) > 0)


def test_rotated_coordinate_follows_beta_law():
    """(Π x)_j of a fixed unit x over many seeds: (u+1)/2 ~ Beta((d-1)/2, (d-1)/2)."""
    d = 16
    x = np.ones(d) / np.sqrt(d)
    samples = []
    for s in range(3000):
        P = rotation.make_rotation(d, 1000 + s)
        samples.append((P @ x)[3])
    a = (d - 1) / 2.0
    p = stats.kstest((np.array(samples) + 1.0) / 2.0, stats.beta(a, a).cdf).pvalue
    assert p > 1e-3
