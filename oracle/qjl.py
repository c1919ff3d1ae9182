"""Quantized Johnson-Lindenstrauss (QJL) stage (oracle side).

[efficiency] §三 "JL 变换" / "非对称估计器": project with a Gaussian matrix
S ∈ R^{m×d}, keep only the signs of the projected key, project the query in
full, and estimate the inner product as

    Prod(q, k) = √(π/2) / m · ‖k‖₂ · ⟨S q, sign(S k)⟩,

which is unbiased, E[Prod] = ⟨q, k⟩.  [memory-wall] §2 stage 2 applies this
1-bit stage to the residual of the MSE stage, so in TurboQuant k is replaced
by r = x - x̃ and ‖k‖ by ‖r‖.

Reading taken where the pages are silent: S has iid N(0, 1) entries (the
√(π/2)/m constant is the unbiasing factor for exactly that law), drawn from
its own seed; sign(0) = +1.

Parity: pinned by Monte-Carlo unbiasedness over ≥ 10^4 independent S and by
the closed-form variance ((π/2)‖q‖²‖r‖² - ⟨q, r⟩²) / m.
"""

import math

import numpy as np

from .prng import gaussian_matrix


def make_qjl(m: int, d: int, seed: int) -> np.ndarray:
    """S (m x d, float64), iid N(0, 1), row-major fill from stream ``seed``."""
    return gaussian_matrix(seed, m, d)


def qjl_alpha(m: int) -> float:
    """√(π/2) / m."""
    return math.sqrt(math.pi / 2.0) / m


def signs(S: np.ndarray, r: np.ndarray) -> np.ndarray:
    """sign(S r) as ±1.0, with sign(0) = +1."""
    p = S @ r
    return np.where(p >= 0.0, 1.0, -1.0)


def estimate(S: np.ndarray, q: np.ndarray, r_norm: float, sigma: np.ndarray) -> float:
    """√(π/2)/m · ‖r‖ · ⟨S q, σ⟩ for stored signs σ (±1)."""
    return qjl_alpha(S.shape[0]) * r_norm * float((S @ q) @ sigma)
