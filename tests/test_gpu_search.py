"""GPU parity of tq_search_topk against the float64 oracle on the same records.

The oracle scores every stored vector with the estimator written as an
explicit reconstruction and sorts.  The GPU accumulates the same estimator in
fp32, so two candidates whose scores differ by less than the fp32 rounding
may swap places; the rule below compares what is unique (well-separated
ranks) and checks that the rest is a valid top-k.
"""

import numpy as np
import pytest
import torch

from oracle import search as osearch
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_generic, make_generic_queries

from parity import gpu_records_to_numpy, oracle_tables, plan

pytestmark = pytest.mark.gpu

REL = 1e-4  # of the largest |score| of the query


def _check_topk(gidx, gsc, osc, k):
    nq, N = osc.shape
    for qi in range(nq):
        s = osc[qi]
        scale = np.abs(s).max()
        tol = REL * scale
        ids = gidx[qi]
        assert len(set(ids.tolist())) == k and ids.min() >= 0 and ids.max() < N
        assert np.all(np.abs(gsc[qi] - s[ids]) <= tol), "returned scores differ from the oracle's"
        assert np.all(np.diff(gsc[qi]) <= 0), "not in descending order"
        order = np.argsort(-s, kind="stable")
        kth = s[order[k - 1]]
        assert np.all(s[ids] >= kth - 2 * tol), "a returned vector is not in the oracle's top-k"
        nxt = s[order[k]] if k < N else -np.inf
        sure = order[:k][s[order[:k]] > nxt + 2 * tol]
        assert set(sure.tolist()) <= set(ids.tolist()), "a clear top-k vector is missing"
        # ranks whose neighbours are well separated agree exactly
        for r in range(k):
            lo = s[order[r + 1]] if r + 1 < N else -np.inf
            hi = s[order[r - 1]] if r > 0 else np.inf
            if s[order[r]] - lo > 2 * tol and hi - s[order[r]] > 2 * tol:
                assert ids[r] == order[r]


def _run(X, Q, d, m, w, k):
    p = plan(d, m, w)
    n = X.shape[0]
    rec = _lib.Records(n, d, m, w)
    _lib.tq_quantize(p, X, rec)
    nq = Q.shape[0]
    ws = torch.empty(_lib.tq_search_workspace_size(p, nq, n, k), dtype=torch.uint8, device="cuda")
    idx = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty(nq, k, device="cuda")
    _lib.tq_search_topk(p, Q, rec, n, k, idx, sc, ws)
    torch.cuda.synchronize()
    got = gpu_records_to_numpy(rec, slice(0, n), d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    osc = osearch.scores(Q.float().cpu().numpy(), got, Pi, S, c)
    return idx.cpu().numpy(), sc.cpu().numpy(), osc


@pytest.mark.parametrize("w", [1, 2, 3])
def test_ragged_sizes_d128(gpu_lib, w):
    g = torch.Generator().manual_seed(100 + w)
    n, nq, k = 9001, 37, 10
    X = torch.randn(n, 128, generator=g) * (1 + 9 * (torch.rand(128, generator=g) < 0.03))
    Q = torch.randn(nq, 128, generator=g)
    gidx, gsc, osc = _run(X.cuda(), Q.cuda(), 128, 128, w, k)
    _check_topk(gidx, gsc, osc, k)


def test_k_equals_n_and_k_64(gpu_lib):
    g = torch.Generator().manual_seed(7)
    X = torch.randn(64, 128, generator=g)
    Q = torch.randn(3, 128, generator=g).to(torch.bfloat16)
    gidx, gsc, osc = _run(X.cuda(), Q.cuda(), 128, 128, 2, 64)
    _check_topk(gidx, gsc, osc, 64)


@pytest.mark.parametrize("d", [128, 96])
def test_k_beyond_n_pads_with_minus_one(gpu_lib, d):
    """k > n: the n stored vectors in rank order, then index -1 and score -inf
    (d = 128 on the tensor-core scores, d = 96 on the SIMT scores)."""
    g = torch.Generator().manual_seed(11 + d)
    n, k = 5, 12
    X = torch.randn(n, d, generator=g)
    Q = torch.randn(3, d, generator=g)
    gidx, gsc, osc = _run(X.cuda(), Q.cuda(), d, d, 2, k)
    _check_topk(gidx[:, :n], gsc[:, :n], osc, n)
    assert np.all(gidx[:, n:] == -1) and np.all(gsc[:, n:] == -np.inf)


def test_generic_d1024_slice(gpu_lib):
    """Unit-norm anisotropic vectors, d = m = 1024, b = 4: 65536 stored, 64 queries, top-10."""
    wl = WORKLOADS["generic"]
    X = make_generic(wl, n=65536, device="cuda")
    Q = make_generic_queries(wl, nq=64, device="cuda")
    gidx, gsc, osc = _run(X, Q, 1024, 1024, 3, 10)
    _check_topk(gidx, gsc, osc, 10)


def test_generic_d1024_full_size(gpu_lib):
    """The generic configuration at its full size: 1,048,576 unit-norm anisotropic vectors,
    d = m = 1024, b = 4, top-10 for 8 queries.  The oracle scores the GPU's records in
    chunks of 65,536."""
    wl = WORKLOADS["generic"]
    n, nq, k, d, m, w = 1 << 20, 8, 10, 1024, 1024, 3
    X = make_generic(wl, n=n, device="cuda")
    Q = make_generic_queries(wl, nq=nq, device="cuda")
    p = plan(d, m, w)
    rec = _lib.Records(n, d, m, w)
    _lib.tq_quantize(p, X, rec)
    del X
    ws = torch.empty(_lib.tq_search_workspace_size(p, nq, n, k), dtype=torch.uint8, device="cuda")
    idx = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty(nq, k, device="cuda")
    _lib.tq_search_topk(p, Q, rec, n, k, idx, sc, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    Pi, S, cent, _ = oracle_tables(d, m, w)
    Qn = Q.float().cpu().numpy()
    osc = np.empty((nq, n))
    step = 1 << 16
    for r0 in range(0, n, step):
        got = gpu_records_to_numpy(rec, slice(r0, r0 + step), d, m, w)
        osc[:, r0:r0 + step] = osearch.scores(Qn, got, Pi, S, cent)
    _check_topk(idx.cpu().numpy(), sc.cpu().numpy(), osc, k)


def test_d512_w1_partial_query_tiles(gpu_lib):
    """d = m = 512, b = 2 (w = 1), 5000 stored vectors, 40 queries (a partial 32-query tile), top-10."""
    g = torch.Generator().manual_seed(512)
    X = torch.randn(5000, 512, generator=g)
    Q = torch.randn(40, 512, generator=g)
    gidx, gsc, osc = _run(X.cuda(), Q.cuda(), 512, 512, 1, 10)
    _check_topk(gidx, gsc, osc, 10)
