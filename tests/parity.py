"""Shared helpers of the GPU parity tests: oracle tables, record conversion and
the comparison rules.

Comparison rules (the method fixes the index rule; the others follow from the
fp32 arithmetic of the kernels):

* indices: at least 99.99 % of coordinates equal; every mismatch is an
  adjacent cell and the oracle's rotated unit coordinate lies within 1e-5 of
  the boundary between the two cells.
* signs: compared on vectors whose indices all match (a different index
  changes the whole residual); at least 99.99 % equal and every flip has
  |(S r)_j| <= 1e-5 · √d · ||r|| (the fp32 rounding of S Πᵀ ρ is far below).
* norms: fp32 norm within 4e-7 relative (fp32 sum of squares vs float64
  rounded once); residual norm within 1e-4 relative on vectors whose
  indices match (u carries ~1e-7 absolute error, ||ρ|| ~ 0.2-0.6).
* scores and attention outputs on the same records: relative L2 error <= 1e-3.
"""

import numpy as np
import torch

from oracle import codebook as ocb
from oracle import pack as opack
from oracle import qjl as oqjl
from oracle import quantize as oquant
from oracle import rotation as orot
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED

_TABLES = {}


def oracle_tables(d, m, w):
    key = (d, m, w)
    if key not in _TABLES:
        Pi = orot.make_rotation(d, ROTATION_SEED)
        S = oqjl.make_qjl(m, d, QJL_SEED)
        c, b, _, _ = ocb.lloyd_max(d, w)
        _TABLES[key] = (Pi, S, c, b)
    return _TABLES[key]


_PLANS = {}


def plan(d, m, w):
    key = (d, m, w)
    if key not in _PLANS:
        _PLANS[key] = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    return _PLANS[key]


def oracle_quantize(X, d, m, w):
    """The oracle's records; m = 0 is stage 1 alone (no QJL rows)."""
    Pi, S, c, b = oracle_tables(d, m, w)
    if m == 0:
        return oquant.quantize_mse(np.asarray(X, dtype=np.float64), Pi, c, b)
    return oquant.quantize(np.asarray(X, dtype=np.float64), Pi, S, c, b)


def gpu_records_to_numpy(rec, rows, d, m, w):
    """Unpack rows of a GPU Records object with the oracle's unpacker (either layout)."""
    if m == 0:  # stage-1-only records: no sign words, no residual norms
        if getattr(rec, "layout", _lib.TQ_LAYOUT_ROWS) == _lib.TQ_LAYOUT_ROWS:
            idx_w = rec.idx[rows].cpu().numpy().view(np.uint32)
            idx = opack.unpack_indices(idx_w, w, d)
            norm = rec.norm[rows].cpu().numpy()
        else:
            r = np.arange(rec.capacity)[rows] if isinstance(rows, slice) else np.asarray(rows)
            b0, b1 = int(r.min()) // 32, int(r.max()) // 32 + 1
            iw = rec.idx.reshape(-1)[b0 * 32 * (w * d // 32):b1 * 32 * (w * d // 32)].cpu().numpy().view(np.uint32)
            idx = opack.unpack_indices_block32(iw.reshape(b1 - b0, w * d), w, d)[r - 32 * b0]
            norm = rec.norm[torch.as_tensor(r)].cpu().numpy()
        n = idx.shape[0]
        return {"idx": idx, "sgn": np.zeros((n, 0), dtype=bool), "norm": norm, "rnorm": np.zeros(n, np.float32),
                "idx_words": opack.pack_indices(idx, w), "sgn_words": np.zeros((n, 0), np.uint32)}
    if getattr(rec, "layout", _lib.TQ_LAYOUT_ROWS) == _lib.TQ_LAYOUT_ROWS:
        idx_w = rec.idx[rows].cpu().numpy().view(np.uint32)
        sgn_w = rec.sgn[rows].cpu().numpy().view(np.uint32)
        return {"idx": opack.unpack_indices(idx_w, w, d), "sgn": opack.unpack_signs(sgn_w),
                "norm": rec.norm[rows].cpu().numpy(), "rnorm": rec.rnorm[rows].cpu().numpy(),
                "idx_words": idx_w, "sgn_words": sgn_w}
    # block layout: unpack whole blocks, then pick the rows
    rows = np.arange(rec.capacity)[rows] if isinstance(rows, slice) else np.asarray(rows)
    b0, b1 = int(rows.min()) // 32, int(rows.max()) // 32 + 1
    iw = rec.idx.reshape(-1)[b0 * 32 * (w * d // 32):b1 * 32 * (w * d // 32)].cpu().numpy().view(np.uint32)
    sw = rec.sgn.reshape(-1)[b0 * 32 * (m // 32):b1 * 32 * (m // 32)].cpu().numpy().view(np.uint32)
    idx = opack.unpack_indices_block32(iw.reshape(b1 - b0, w * d), w, d)[rows - 32 * b0]
    sgn = opack.unpack_signs_block32(sw.reshape(b1 - b0, m))[rows - 32 * b0]
    return {"idx": idx, "sgn": sgn, "norm": rec.norm[torch.as_tensor(rows)].cpu().numpy(),
            "rnorm": rec.rnorm[torch.as_tensor(rows)].cpu().numpy(),
            "idx_words": opack.pack_indices(idx, w), "sgn_words": opack.pack_signs(sgn)}


def oracle_records_to_gpu(q, d, m, w, device="cuda", layout=None):
    """Pack an oracle Quantized result with the oracle's packer and upload it."""
    layout = _lib.TQ_LAYOUT_ROWS if layout is None else layout
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    if m == 0:  # stage-1-only records: indices and norms
        n = q.idx.shape[0]
        idx_w = (opack.pack_indices(q.idx, w) if layout == _lib.TQ_LAYOUT_ROWS else
                 opack.pack_indices_block32(q.idx, w).reshape(n, w * d // 32)).view(np.int32)
        return _lib.Records.wrap(t(idx_w), None, t(q.norm), None, d, m, w, layout=layout)
    if layout == _lib.TQ_LAYOUT_ROWS:
        idx_w = opack.pack_indices(q.idx, w).view(np.int32)
        sgn_w = opack.pack_signs(q.sgn).view(np.int32)
    else:
        n = q.idx.shape[0]
        idx_w = opack.pack_indices_block32(q.idx, w).reshape(n, w * d // 32).view(np.int32)
        sgn_w = opack.pack_signs_block32(q.sgn).reshape(n, m // 32).view(np.int32)
    return _lib.Records.wrap(t(idx_w), t(sgn_w), t(q.norm), t(q.rnorm), d, m, w, layout=layout)


def check_indices(got_idx, oq, bounds, min_match=0.9999, tol=1e-5):
    """Index rule; returns the boolean mask of fully matching vectors."""
    eq = got_idx == oq.idx
    frac = eq.mean()
    assert frac >= min_match, f"index match {frac:.6f} < {min_match}"
    bad = np.argwhere(~eq)
    for v, j in bad:
        a, b = sorted((int(got_idx[v, j]), int(oq.idx[v, j])))
        assert b - a == 1, f"non-adjacent cells {a}, {b} at ({v}, {j})"
        assert abs(oq.u[v, j] - bounds[a]) <= tol, f"mismatch {abs(oq.u[v, j] - bounds[a])} from boundary"
    return eq.all(axis=1)


def check_signs(got_sgn, oq, rows_ok, d, min_match=0.9999):
    g = got_sgn[rows_ok]
    o = oq.sgn[rows_ok]
    if g.size == 0:
        return
    eq = g == o
    assert eq.mean() >= min_match, f"sign match {eq.mean():.6f}"
    p = oq.p[rows_ok]
    rn = oq.rnorm64[rows_ok][:, None] * np.ones_like(p)
    flips = ~eq
    assert np.all(np.abs(p[flips]) <= 1e-5 * np.sqrt(d) * rn[flips]), "sign flip away from zero"


def check_norms(got, oq, rows_ok):
    n64 = oq.norm.astype(np.float64)
    assert np.all(np.abs(got["norm"] - n64) <= 4e-7 * np.abs(n64) + 1e-30)
    r64 = oq.rnorm64[rows_ok]
    assert np.all(np.abs(got["rnorm"][rows_ok] - r64) <= 1e-4 * r64 + 1e-30)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)
