"""Random rotation Π (oracle side).

[memory-wall] §2 stage 1 and [efficiency] §四 Step 1 ("Random
Preconditioning"): each vector is multiplied by one fixed random orthogonal
matrix, which preserves inner products and spreads energy over all
coordinates.  The pages do not fix how Π is drawn; the reading taken here is
the Haar construction: G with iid N(0, 1) entries, G = QR, Π = Q·diag(sign
diag R), i.e. the unique QR factor whose R has a positive diagonal.  The
convention is u = Π x (rows of Π are the new basis).

Parity: pinned by ΠΠᵀ = I, ‖Πx‖ = ‖x‖, Πᵀ G upper triangular with a positive
diagonal, and the Beta coordinate law of Π x (KS test).
"""

import numpy as np

from .prng import gaussian_matrix


def make_rotation(d: int, seed: int) -> np.ndarray:
    """Π (d x d, float64) for stream ``seed``; u = Π @ x."""
    g = gaussian_matrix(seed, d, d)
    q, r = np.linalg.qr(g)
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]
