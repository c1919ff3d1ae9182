"""GPU parity of the tcgen05 search (d a multiple of 256 up to 1024, m = d or 0,
k <= 16) against the float64 oracle's scores of the same records.

The kernel forms the estimator of "TurboQuant 与 AI 效率革命" §三 over 128
queries x 256 stored vectors per tensor-core unit and keeps each query's best
per CTA; the top-k rule of tests/test_gpu_search.py decides (returned scores
within 1e-4 of the query's largest |score|, a valid top-k, well-separated
ranks in the oracle's order).  Cases cover every w, ragged query blocks and
vector units, several units per CTA, k = 1 and k = 16, k beyond the path
(17: the warp-MMA kernel), k > n, and zero norms.
"""

import numpy as np
import pytest
import torch

from oracle import search as osearch
from online_kv_cache_04_b300 import _lib

from parity import gpu_records_to_numpy, oracle_tables, plan
from test_gpu_search import _check_topk

pytestmark = pytest.mark.gpu


def _search(X, Q, d, m, w, k):
    p = plan(d, m, w)
    n, nq = X.shape[0], Q.shape[0]
    rec = _lib.Records(n, d, m, w)
    _lib.tq_quantize(p, X, rec)
    ws = torch.empty(_lib.tq_search_workspace_size(p, nq, n, k), dtype=torch.uint8, device="cuda")
    idx = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty(nq, k, device="cuda")
    _lib.tq_search_topk(p, Q, rec, n, k, idx, sc, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags(reset=True) == 0
    got = gpu_records_to_numpy(rec, slice(0, n), d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    osc = osearch.scores(Q.float().cpu().numpy(), got, Pi, S, c, qjl_stage=m > 0)
    return idx.cpu().numpy(), sc.cpu().numpy(), osc


def _data(n, nq, d, seed):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(n, d, generator=g) * (1 + 9 * (torch.rand(d, generator=g) < 0.03))
    Q = torch.randn(nq, d, generator=g)
    return X.cuda(), Q.cuda()


@pytest.mark.parametrize("d", [256, 512, 1024])
@pytest.mark.parametrize("w", [1, 2, 3])
def test_two_stage_ragged_blocks(gpu_lib, d, w):
    """3001 stored vectors (the last 256-vector unit partial), 130 queries (two
    128-query blocks, the second with 2), top-10."""
    X, Q = _data(3001, 130, d, 8000 + d + w)
    gidx, gsc, osc = _search(X, Q, d, d, w, 10)
    _check_topk(gidx, gsc, osc, 10)


@pytest.mark.parametrize("k", [1, 16, 17])
def test_list_lengths(gpu_lib, k):
    """k = 1 and the longest list the path keeps (16); 17 takes the warp-MMA kernel."""
    X, Q = _data(5000, 24, 512, 8100 + k)
    gidx, gsc, osc = _search(X, Q, 512, 512, 3, k)
    _check_topk(gidx, gsc, osc, k)


def test_many_units_per_cta(gpu_lib):
    """100,003 stored vectors and 200 queries at d = 256: two query blocks, so 74
    CTAs per block each walk five or six units."""
    X, Q = _data(100003, 200, 256, 8200)
    gidx, gsc, osc = _search(X, Q, 256, 256, 2, 10)
    _check_topk(gidx, gsc, osc, 10)


def test_k_beyond_n_and_zero_vectors(gpu_lib):
    """k > n pads with index -1 and score -inf; zero vectors (zero norms) score 0."""
    X, Q = _data(6, 3, 256, 8300)
    X[2] = 0.0
    k = 12
    gidx, gsc, osc = _search(X, Q, 256, 256, 3, k)
    _check_topk(gidx[:, :6], gsc[:, :6], osc, 6)
    assert np.all(gidx[:, 6:] == -1) and np.all(gsc[:, 6:] == -np.inf)


@pytest.mark.parametrize("w", [1, 3])
def test_stage1_alone(gpu_lib, w):
    """m = 0: the codebook part alone ("谷歌TurboQuant如何绕过内存墙？" §2 stage 1)."""
    X, Q = _data(4000, 33, 512, 8400 + w)
    gidx, gsc, osc = _search(X, Q, 512, 0, w, 10)
    _check_topk(gidx, gsc, osc, 10)
