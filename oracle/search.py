"""Inner-product top-k search over compressed vectors (oracle side).

[video] and [memory-wall] name vector search engines as the second use of
the same quantizer.  The score of stored vector i for query q is the same
unbiased estimator as in attention, without the softmax scale:
⟨q, x̃_i⟩ + √(π/2)/m · ‖r_i‖ · ⟨S q, σ_i⟩ = ⟨q, x̂_i⟩.  The k largest scores
are returned in descending order; equal scores go to the lower index.

Parity: pinned by the exact-codeword special case (then the result is plain
exhaustive maximum-inner-product search) and by brute force on tiny sets.
"""

import numpy as np

from .quantize import reconstruct


def scores(Q, rec, Pi, S, centroids, qjl_stage=True):
    """[nq, N] estimated inner products (stage 1 alone when qjl_stage is False)."""
    xh = reconstruct(rec["idx"], rec["sgn"], rec["norm"], rec["rnorm"], Pi, S, centroids, qjl_stage=qjl_stage)
    return np.asarray(Q, dtype=np.float64) @ xh.T


def topk(Q, rec, Pi, S, centroids, k, qjl_stage=True):
    """(indices [nq, k] int64, scores [nq, k] float64)."""
    sc = scores(Q, rec, Pi, S, centroids, qjl_stage=qjl_stage)
    order = np.argsort(-sc, axis=1, kind="stable")[:, :k]
    return order, np.take_along_axis(sc, order, axis=1)
