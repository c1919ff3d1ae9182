"""Outlier-channel split precision (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"TurboQuant压缩效果" (douyin transcripts), the part on 2.5 and 3.5 bits: the
128 channels of a head are split; a few especially important outlier channels
get 3 bits and the ordinary ones 2, and "2.5 bits" is the average over the
channels (3.5 bits likewise, one bit higher).

Reading taken (the page gives no sizes and no procedure):

* A head's d channels are split by a fixed permutation ``perm``: the n_o
  outlier channels perm[:n_o] and the d - n_o regular channels perm[n_o:].
  The split is a property of the head, fixed before any vector is quantized
  (no calibration of the quantizer itself).  ``choose_outliers`` gives one
  data-free-of-tuning choice: the n_o channels with the largest mean square
  over a sample of the head's vectors, lowest channel first on ties.
* The split happens before the rotation (a rotation of all d channels would
  spread the outliers over every coordinate).  Each side is quantized by its
  own TurboQuant instance ([memory-wall] §2 stages 1 and 2): its own rotation
  of its own dimension, the Lloyd-Max codebook of its own coordinate law
  f_{n_o} or f_{d - n_o}, its own QJL matrix with as many rows as channels,
  its own fp32 norm and residual norm.  Outliers take b_R + 1 total bits,
  regular channels b_R (each total = MSE bits + the 1 QJL bit).
* Inner products split over the channel sets, ⟨q, k⟩ = ⟨q_O, k_O⟩ +
  ⟨q_R, k_R⟩, so a score is the sum of the two instances' estimators, and a
  reconstructed vector carries each instance's reconstruction at its channels.
* Bits per coordinate of indices and signs: (n_o (b_R + 1) + (d - n_o) b_R)/d
  = b_R + n_o/d.  The page's labels 2.5 and 3.5 are b_R = 2 and 3 with
  n_o = d/2 (the average it states holds only with half the channels
  promoted, although it calls them "a few"); the four fp32 norms add 128/d
  bits per coordinate.

Parity: pinned by the bit accounting at the page's labels, exact
reconstruction of vectors that lie on a codeword ray of both instances,
Monte-Carlo unbiasedness of the split score over independent QJL matrices,
the expected stage-1 distortion of each side from its own codebook's MSE,
and recovery of planted outlier channels.
"""

from dataclasses import dataclass

import numpy as np

from . import codebook, qjl, quantize, rotation


@dataclass
class SplitTables:
    """The two instances' tables: outliers (O) and regular channels (R)."""
    perm: np.ndarray     # [d] int64: perm[:n_o] outlier channels, perm[n_o:] the rest
    n_o: int
    Pi_O: np.ndarray     # [n_o, n_o]
    S_O: np.ndarray      # [n_o, n_o]
    c_O: np.ndarray      # centroids, 2^(b_R) levels
    b_O: np.ndarray      # bounds
    Pi_R: np.ndarray     # [d - n_o, d - n_o]
    S_R: np.ndarray
    c_R: np.ndarray      # 2^(b_R - 1) levels
    b_R: np.ndarray


def choose_outliers(X_sample: np.ndarray, n_o: int) -> np.ndarray:
    """perm for the n_o channels of largest mean square over the sample rows
    (ties -> lower channel), outliers then the rest, each ascending."""
    X = np.asarray(X_sample, dtype=np.float64)
    ms = np.mean(X * X, axis=0)
    d = ms.shape[0]
    order = sorted(range(d), key=lambda j: (-ms[j], j))
    out = np.array(sorted(order[:n_o]), dtype=np.int64)
    rest = np.array(sorted(order[n_o:]), dtype=np.int64)
    return np.concatenate([out, rest])


def make_tables(perm, n_o: int, bits_regular: int, rot_seed_O: int, qjl_seed_O: int, rot_seed_R: int,
                qjl_seed_R: int) -> SplitTables:
    """Tables of the two instances: outliers at bits_regular + 1 total bits
    (bits_regular MSE bits), the rest at bits_regular (bits_regular - 1 MSE bits)."""
    perm = np.asarray(perm, dtype=np.int64)
    d = perm.shape[0]
    d_R = d - n_o
    c_O, bo, _, _ = codebook.lloyd_max(n_o, bits_regular)
    c_R, br, _, _ = codebook.lloyd_max(d_R, bits_regular - 1)
    return SplitTables(perm=perm, n_o=n_o,
                       Pi_O=rotation.make_rotation(n_o, rot_seed_O), S_O=qjl.make_qjl(n_o, n_o, qjl_seed_O),
                       c_O=c_O, b_O=bo,
                       Pi_R=rotation.make_rotation(d_R, rot_seed_R), S_R=qjl.make_qjl(d_R, d_R, qjl_seed_R),
                       c_R=c_R, b_R=br)


def split(X, t: SplitTables):
    """(X[:, perm[:n_o]], X[:, perm[n_o:]])."""
    X = np.asarray(X, dtype=np.float64)
    return X[:, t.perm[:t.n_o]], X[:, t.perm[t.n_o:]]


def quantize_split(X, t: SplitTables):
    """The two instances' records (quantize.Quantized each) of the rows of X [N, d]."""
    XO, XR = split(X, t)
    return (quantize.quantize(XO, t.Pi_O, t.S_O, t.c_O, t.b_O),
            quantize.quantize(XR, t.Pi_R, t.S_R, t.c_R, t.b_R))


def reconstruct_split(qO, qR, t: SplitTables, qjl_stage: bool = True) -> np.ndarray:
    """x̂ [N, d]: each instance's unbiased reconstruction at its own channels."""
    xO = quantize.reconstruct(qO.idx, qO.sgn, qO.norm, qO.rnorm, t.Pi_O, t.S_O, t.c_O, qjl_stage)
    xR = quantize.reconstruct(qR.idx, qR.sgn, qR.norm, qR.rnorm, t.Pi_R, t.S_R, t.c_R, qjl_stage)
    out = np.empty((xO.shape[0], t.perm.shape[0]))
    out[:, t.perm[:t.n_o]] = xO
    out[:, t.perm[t.n_o:]] = xR
    return out


def score_split(q, qO, qR, t: SplitTables) -> np.ndarray:
    """Estimated ⟨q, x_i⟩ for every stored row i: the sum of the two instances'
    estimators ⟨q_part, x̃_part⟩ + √(π/2)/m_part ‖r_part‖ ⟨S_part q_part, σ_part⟩."""
    q = np.asarray(q, dtype=np.float64)
    total = np.zeros(qO.idx.shape[0])
    for qq, Pi, S, c, ch in ((qO, t.Pi_O, t.S_O, t.c_O, t.perm[:t.n_o]), (qR, t.Pi_R, t.S_R, t.c_R, t.perm[t.n_o:])):
        qp = q[ch]
        stage1 = np.asarray(qq.norm, dtype=np.float64) * (c[qq.idx] @ (Pi @ qp))
        sig = np.where(qq.sgn, 1.0, -1.0)
        total += stage1 + qjl.qjl_alpha(S.shape[0]) * np.asarray(qq.rnorm, dtype=np.float64) * (sig @ (S @ qp))
    return total


def bits_per_coordinate(d: int, n_o: int, bits_regular: int, with_norms: bool = False) -> float:
    """(n_o (b_R + 1) + (d - n_o) b_R) / d, plus the four fp32 norms if asked."""
    bits = n_o * (bits_regular + 1) + (d - n_o) * bits_regular
    if with_norms:
        bits += 4 * 32
    return bits / d


def decode_attention_split(q, K_O, K_R, V_O, V_R, ctx_len, t: SplitTables, scale=None, t_v: SplitTables = None):
    """Softmax attention over split records.  q [B, Hq, d]; each record dict as
    in decode.reconstruct_cache ([B, Hkv, T, ...]); the cache reconstructions are
    assembled channel by channel (keys with t, values with t_v, default t) and
    then attended exactly as decode.attention."""
    t_v = t if t_v is None else t_v
    from .decode import attention

    def recon(RO, RR, t):
        lead = RO["idx"].shape[:-1]
        n = int(np.prod(lead))
        flat = lambda R, k, last: R[k].reshape((n,) + ((last,) if last is not None else ()))
        qO = quantize.Quantized(idx=flat(RO, "idx", RO["idx"].shape[-1]), sgn=flat(RO, "sgn", RO["sgn"].shape[-1]),
                                norm=flat(RO, "norm", None), rnorm=flat(RO, "rnorm", None), u=None, p=None,
                                rnorm64=None)
        qR = quantize.Quantized(idx=flat(RR, "idx", RR["idx"].shape[-1]), sgn=flat(RR, "sgn", RR["sgn"].shape[-1]),
                                norm=flat(RR, "norm", None), rnorm=flat(RR, "rnorm", None), u=None, p=None,
                                rnorm64=None)
        return reconstruct_split(qO, qR, t).reshape(lead + (t.perm.shape[0],))

    return attention(q, recon(K_O, K_R, t), recon(V_O, V_R, t_v), ctx_len, scale)
