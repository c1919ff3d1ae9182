"""The two-stage TurboQuant vector quantizer (oracle side).

Steps, in the order of [memory-wall] §2 and [efficiency] §四:

1. n = ‖x‖₂, stored as one fp32 ([efficiency] §三 "零开销的秘密": one 32-bit
   norm per vector).  u = Π x / n is a point on the unit sphere whose
   coordinates follow f_d.
2. Stage 1, (b-1) = w bits per coordinate: idx_j = #{k : β_k < u_j}, the
   Lloyd-Max cell of u_j (a tie goes to the lower cell).  Reconstruction
   x̃ = n · Πᵀ c[idx].  No scale or zero point is stored.
3. Stage 2, 1 bit per JL row: residual r = x - x̃ in the original domain,
   p = S r, σ_j = sign(p_j) with sign(0) = +1; ‖r‖₂ stored as fp32.

Zero vector: n = 0 gives u = 0 (bucketized by the tie rule), r = 0 and all
σ = +1.  Inputs are taken exactly into float64; the two norms are rounded to
fp32 (round to nearest even) only when stored.

Parity: pinned through the codebook and QJL pins, brute-force nearest
codeword search on d = 8, the exact-codeword special case (r = 0), the
printed MSE bounds and the 2/π bias of the 1-bit MSE quantizer.
"""

from dataclasses import dataclass

import numpy as np


@dataclass
class Quantized:
    idx: np.ndarray      # [N, d] int64 in [0, 2^w)
    sgn: np.ndarray      # [N, m] bool, True <-> σ = +1
    norm: np.ndarray     # [N] float32, fp32(‖x‖)
    rnorm: np.ndarray    # [N] float32, fp32(‖r‖)
    u: np.ndarray        # [N, d] float64 rotated unit coordinates (diagnostic)
    p: np.ndarray        # [N, m] float64 S r (diagnostic)
    rnorm64: np.ndarray  # [N] float64 ‖r‖ (diagnostic)


def bucketize(u: np.ndarray, bounds: np.ndarray) -> np.ndarray:
    """idx = #{k : β_k < u} for every element (tie -> lower cell)."""
    return np.searchsorted(bounds, u, side="left").astype(np.int64)


def stage1(X: np.ndarray, Pi: np.ndarray, centroids: np.ndarray, bounds: np.ndarray):
    """Stage 1 only: returns (n, u, idx, x̃)."""
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=1))
    safe = np.where(n > 0.0, n, 1.0)
    u = (X @ Pi.T) / safe[:, None]
    u[n == 0.0] = 0.0
    idx = bucketize(u, bounds)
    xt = n[:, None] * (centroids[idx] @ Pi)  # rows: n · Πᵀ c[idx]
    return n, u, idx, xt


def quantize(X: np.ndarray, Pi: np.ndarray, S: np.ndarray, centroids: np.ndarray,
             bounds: np.ndarray) -> Quantized:
    """Quantize the rows of X [N, d] with Π [d, d], S [m, d] and a codebook."""
    n, u, idx, xt = stage1(X, Pi, centroids, bounds)
    r = np.asarray(X, dtype=np.float64) - xt
    p = r @ S.T
    rn = np.sqrt(np.sum(r * r, axis=1))
    return Quantized(idx=idx, sgn=p >= 0.0, norm=n.astype(np.float32), rnorm=rn.astype(np.float32),
                     u=u, p=p, rnorm64=rn)


def quantize_mse(X: np.ndarray, Pi: np.ndarray, centroids: np.ndarray, bounds: np.ndarray) -> Quantized:
    """Stage 1 alone as the stored format: the rotation and the MSE-optimal
    per-coordinate codebook with every bit of the budget ([memory-wall] §2
    stage 1), stored as (idx, fp32 ‖x‖) -- no QJL rows,
    no residual norm.  Its reconstruction n · Πᵀ c[idx] is the MSE-optimal one;
    its inner products carry the stage-1 bias (2/π at one bit)."""
    n, u, idx, _ = stage1(X, Pi, centroids, bounds)
    N = idx.shape[0]
    return Quantized(idx=idx, sgn=np.zeros((N, 0), dtype=bool), norm=n.astype(np.float32),
                     rnorm=np.zeros(N, dtype=np.float32), u=u, p=np.zeros((N, 0)), rnorm64=np.zeros(N))


def reconstruct(idx: np.ndarray, sgn: np.ndarray, norm: np.ndarray, rnorm: np.ndarray,
                Pi: np.ndarray, S: np.ndarray, centroids: np.ndarray, qjl_stage: bool = True) -> np.ndarray:
    """Unbiased reconstruction from stored record values.

    x̂ = norm · Πᵀ c[idx] + √(π/2)/m · rnorm · Sᵀ σ.  Its inner product with
    any q is exactly the estimator of [memory-wall] §2 stage 2 / [efficiency]
    §三: ⟨q, x̃⟩ + √(π/2)/m ‖r‖ ⟨S q, σ⟩.
    """
    m = S.shape[0]
    nrm = np.asarray(norm, dtype=np.float64)
    x = nrm[:, None] * (centroids[idx] @ Pi)
    if qjl_stage:
        sig = np.where(sgn, 1.0, -1.0)
        x = x + (np.sqrt(np.pi / 2.0) / m) * np.asarray(rnorm, dtype=np.float64)[:, None] * (sig @ S)
    return x
