"""Lloyd-Max codebook for the post-rotation coordinate law (oracle side).

[memory-wall] §2 stage 1: after a random rotation every coordinate of a unit
vector follows one known Beta-type law, so the MSE-optimal scalar quantizer
(Lloyd-Max: one-dimensional continuous k-means) can be computed once per bit
width and stored; no scale or zero point is kept.  The law of one coordinate
of a uniformly random unit vector in R^d is

    f_d(x) = Γ(d/2) / (√π Γ((d-1)/2)) · (1 - x²)^((d-3)/2),   -1 ≤ x ≤ 1.

Lloyd-Max alternates the two optimality conditions until they hold together:
each boundary is the midpoint of its two neighbouring centroids, and each
centroid is the conditional mean of its cell.  Cell masses come from the
regularized incomplete beta function, P(|X| ≤ t) = I_{t²}(1/2, (d-1)/2);
first moments from the closed form ∫ x (1-x²)^a dx = -(1-x²)^(a+1) / (2(a+1)).
The law is symmetric, so the iteration runs on the positive half and mirrors.

Parity: pinned by the w = 1 closed form c = ±Γ(d/2)/(√π Γ((d+1)/2)), by
independent adaptive quadrature, by the MSE bounds printed in [memory-wall]
§2 (4^-w ≤ d·MSE ≤ (√3·π/2)·4^-w, ratio ≈ 1.45 at w = 1), and by Max's
Gaussian quantizer as d → ∞.
"""

import math

import numpy as np
from scipy import special


def gamma_half_ratio(d: int) -> float:
    """Γ(d/2) / Γ((d-1)/2), from Γ(3/2)/Γ(1) = √π/2, Γ(2)/Γ(3/2) = 2/√π and the
    recurrence ratio(d + 2) = ratio(d) · d / (d - 1) (Γ(x + 1) = x Γ(x)); for
    d > 4096 the classical expansion Γ(x+½)/Γ(x) = √x (1 - 1/(8x) + 1/(128x²)
    + 5/(1024x³) - 21/(32768x⁴) + ...) with x = (d-1)/2."""
    if d > 4096:
        x = (d - 1) / 2.0
        return math.sqrt(x) * (1 - 1 / (8 * x) + 1 / (128 * x ** 2) + 5 / (1024 * x ** 3) - 21 / (32768 * x ** 4))
    r = math.sqrt(math.pi) / 2.0 if d % 2 == 1 else 2.0 / math.sqrt(math.pi)
    for k in range(3 if d % 2 == 1 else 4, d, 2):
        r *= k / (k - 1.0)
    return r


def density_const(d: int) -> float:
    """Normalising constant Γ(d/2) / (√π Γ((d-1)/2)) of f_d."""
    return gamma_half_ratio(d) / math.sqrt(math.pi)


def density(x, d: int):
    """f_d(x) on [-1, 1]."""
    x = np.asarray(x, dtype=np.float64)
    return density_const(d) * np.power(np.clip(1.0 - x * x, 0.0, None), (d - 3) / 2.0)


def _half_mass(a: float, b: float, d: int) -> float:
    """P(a ≤ X ≤ b) for 0 ≤ a ≤ b ≤ 1."""
    bb = (d - 1) / 2.0
    if b >= 1.0:
        return 0.5 * special.betaincc(0.5, bb, a * a)
    return 0.5 * (special.betainc(0.5, bb, b * b) - special.betainc(0.5, bb, a * a))


def _half_moment(a: float, b: float, d: int) -> float:
    """∫_a^b x f_d(x) dx for 0 ≤ a ≤ b ≤ 1 (closed form)."""
    ap1 = (d - 1) / 2.0  # exponent (d-3)/2 plus one
    return density_const(d) * ((1.0 - a * a) ** ap1 - (1.0 - min(b, 1.0) ** 2) ** ap1) / (2.0 * ap1)


def lloyd_max(d: int, w: int, max_iter: int = 20000):
    """Lloyd-Max quantizer with L = 2^w levels for f_d.

    Returns (centroids[L] ascending, bounds[L-1] ascending, mse_per_coord,
    iterations).  mse_per_coord = E[(X - Q(X))²] = 1/d - Σ p_i c_i².
    """
    if d < 3 or w < 1:
        raise ValueError("need d >= 3 and w >= 1")
    half = (1 << w) // 2
    bb = (d - 1) / 2.0
    # start: conditional means of the equal-probability cells of f_d
    qs = [0.0] + [math.sqrt(special.betaincinv(0.5, bb, 2.0 * k / (2 * half))) for k in range(1, half)] + [1.0]
    c = np.array([_half_moment(qs[k], qs[k + 1], d) / _half_mass(qs[k], qs[k + 1], d) for k in range(half)])
    it = 0
    best, since_best = np.inf, 0
    for it in range(1, max_iter + 1):
        t = [0.0] + [0.5 * (c[k] + c[k + 1]) for k in range(half - 1)] + [1.0]
        cn = np.array([_half_moment(t[k], t[k + 1], d) / _half_mass(t[k], t[k + 1], d) for k in range(half)])
        delta = np.max(np.abs(cn - c))
        c = cn
        if delta <= 1e-14 * c[-1]:
            break
        # stop once the step no longer shrinks: the float64 noise floor of the fixed point
        if delta < best:
            best, since_best = delta, 0
        else:
            since_best += 1
            if since_best >= 100 and best <= 1e-12 * c[-1]:
                break
    t = [0.0] + [0.5 * (c[k] + c[k + 1]) for k in range(half - 1)] + [1.0]
    p = np.array([_half_mass(t[k], t[k + 1], d) for k in range(half)])
    mse = 1.0 / d - 2.0 * float(np.sum(p * c * c))
    centroids = np.concatenate([-c[::-1], c])
    pos_bounds = np.array(t[1:-1])
    bounds = np.concatenate([-pos_bounds[::-1], [0.0], pos_bounds])
    return centroids, bounds, mse, it


def codebook_mse_numeric(centroids: np.ndarray, bounds: np.ndarray, d: int) -> float:
    """E[(X - Q(X))²] by adaptive quadrature of f_d (independent of lloyd_max)."""
    from scipy import integrate

    edges = np.concatenate([[-1.0], bounds, [1.0]])
    total = 0.0
    for i, c in enumerate(centroids):
        val, _ = integrate.quad(lambda x: (x - c) ** 2 * density(x, d), edges[i], edges[i + 1],
                                epsabs=1e-15, epsrel=1e-13, limit=400)
        total += val
    return total
