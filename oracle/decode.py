"""Decode attention over the compressed cache (oracle side).

Attention scores are query-key inner products ([memory-wall] §2 stage 2:
biased inner products skew the scores); TurboQuant's estimator of ⟨q, k⟩ from
a stored record is ⟨q, x̃⟩ + √(π/2)/m · ‖r‖ · ⟨S q, σ⟩ ([efficiency] §三
asymmetric estimator, applied to the residual as in [memory-wall] §2).  The
oracle writes that estimator as an explicit reconstruction x̂ (see
``quantize.reconstruct``) and then runs textbook softmax attention:

    s_{g,t} = scale · ⟨q_g, k̂_t⟩,        scale = 1/√d unless given,
    p_{g,·} = softmax over t < ctx_len[b],
    o_g     = Σ_t p_{g,t} v̂_t,

where query head g reads kv head ⌊g / (Hq/Hkv)⌋ (consecutive grouping) and v̂
is the same unbiased reconstruction applied to the value records (reading:
the value side keeps both stages).

Parity: pinned by the exact-codeword special case (records that reconstruct
exactly reduce this to library softmax attention), ctx_len = 1, q = 0 and
token-permutation invariants, and MC unbiasedness of the scores.
"""

import numpy as np

from .quantize import reconstruct


def reconstruct_cache(rec, Pi, S, centroids, qjl_stage=True):
    """rec: dict idx [..., T, d], sgn [..., T, m], norm [..., T], rnorm [..., T]."""
    idx = rec["idx"]
    lead = idx.shape[:-1]
    d = idx.shape[-1]
    m = rec["sgn"].shape[-1]
    n = int(np.prod(lead))  # explicit: a stage-1-only record has m = 0 sign columns
    x = reconstruct(idx.reshape(n, d), rec["sgn"].reshape(n, m), rec["norm"].reshape(n),
                    rec["rnorm"].reshape(n), Pi, S, centroids, qjl_stage=qjl_stage)
    return x.reshape(lead + (d,))


def attention(q, Kh, Vh, ctx_len, scale=None):
    """Softmax attention, float64.  q [B, Hq, d]; Kh, Vh [B, Hkv, T, d]; ctx_len [B].

    Returns (out [B, Hq, d], scores [B, Hq, T] with -inf beyond ctx_len).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = Kh.shape[1]
    T = Kh.shape[2]
    G = Hq // Hkv
    if scale is None or scale == 0.0:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, Hq, d))
    scores = np.full((B, Hq, T), -np.inf)
    for b in range(B):
        L = int(ctx_len[b])
        for g in range(Hq):
            h = g // G
            if L == 0:
                continue
            s = scale * (Kh[b, h, :L] @ q[b, g])
            scores[b, g, :L] = s
            e = np.exp(s - np.max(s))
            p = e / np.sum(e)
            out[b, g] = p @ Vh[b, h, :L]
    return out, scores


def decode_attention(q, K_rec, V_rec, ctx_len, Pi, S, centroids, scale=None, qjl_stage=True):
    """Attention of q over stored K/V records (see module docstring)."""
    Kh = reconstruct_cache(K_rec, Pi, S, centroids, qjl_stage=qjl_stage)
    Vh = reconstruct_cache(V_rec, Pi, S, centroids, qjl_stage=qjl_stage)
    return attention(q, Kh, Vh, ctx_len, scale)
