"""GPU parity of stage-1-only plans (m = 0) against the float64 oracle.

A plan without QJL rows stores the rotation and the MSE-optimal codebook
index of every coordinate plus the fp32 norm ("谷歌TurboQuant如何绕过内存墙？"
§2 stage 1 used alone, with all w bits).  The library runs such plans on its
general kernels; these tests hold them to the same rules as the two-stage
records: the index rule of tests/parity.py, fp32 norms, relative L2 <= 1e-3
for attention outputs, and the search top-k rule.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from oracle import search as osearch
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_generic, make_generic_queries, make_kv

from parity import (check_indices, check_norms, gpu_records_to_numpy, oracle_quantize, oracle_records_to_gpu,
                    oracle_tables, plan, rel_l2)
from test_gpu_search import _check_topk

pytestmark = pytest.mark.gpu
BLK = _lib.TQ_LAYOUT_BLOCK32


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("d,dtype,layout,n,off", [(128, torch.float32, 0, 1000, 0),
                                                   (128, torch.bfloat16, 0, 777, 5),
                                                   (128, torch.bfloat16, 1, 1000, 64),
                                                   (256, torch.float32, 1, 300, 20)])
def test_quantize_stage1_only(gpu_lib, w, d, dtype, layout, n, off):
    wl = WORKLOADS["llama8b"]
    X = make_kv(wl, B=1, T=n, which=0, device="cuda")[0, 0].to(dtype)
    if d != 128:
        X = torch.cat([X, X.flip(1)], dim=1).contiguous()
    p = plan(d, 0, w)
    cap = (n + off + 63) // 32 * 32
    rec = _lib.Records(cap, d, 0, w, layout=layout)
    rec.idx.fill_(-1)
    _lib.tq_quantize(p, X, rec, out_offset=off)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    oq = oracle_quantize(X.float().cpu().numpy(), d, 0, w)
    got = gpu_records_to_numpy(rec, slice(off, off + n), d, 0, w)
    _, _, _, bounds = oracle_tables(d, 0, w)
    ok = check_indices(got["idx"], oq, bounds)
    check_norms(got, oq, ok)


@pytest.mark.parametrize("w", [1, 2, 3])
def test_quantize_pair_stage1_only_equals_two_calls(gpu_lib, w):
    d = 128
    wl = WORKLOADS["llama8b"]
    K = make_kv(wl, B=1, T=640, which=0, device="cuda")[0, 0].contiguous()
    V = make_kv(wl, B=1, T=640, which=1, device="cuda")[0, 0].contiguous()
    p = plan(d, 0, w)
    outs = []
    for pair in (True, False):
        rk, rv = _lib.Records(640, d, 0, w), _lib.Records(640, d, 0, w, layout=BLK)
        if pair:
            _lib.tq_quantize_pair(p, K, V, rk, rv)
        else:
            _lib.tq_quantize(p, K, rk)
            _lib.tq_quantize(p, V, rv)
        torch.cuda.synchronize()
        outs.append([t.cpu().numpy() for t in (rk.idx, rk.norm, rv.idx, rv.norm)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("vlayout,Hq,T,ctx", [(0, 8, 640, [640, 333]), (1, 8, 640, [640, 333]),
                                              (1, 16, 1152, [1152, 1]), (1, 4, 9216, [9216, 5000])])
def test_decode_stage1_only_oracle_records(gpu_lib, w, vlayout, Hq, T, ctx):
    """GQA 4 : 2 to 16 : 2 over two batch rows of ragged length, on the oracle's own
    records; values by row take the general kernels, values in blocks the warp-MMA
    kernel (9216 tokens span many tiles and CTAs)."""
    d = 128
    B, Hkv = 2, 2
    g = torch.Generator().manual_seed(70 + w + T)
    K = torch.randn(B, Hkv, T, d, generator=g)
    V = torch.randn(B, Hkv, T, d, generator=g)
    q = torch.randn(B, Hq, d, generator=g)
    kq = oracle_quantize(K.reshape(-1, d).numpy(), d, 0, w)
    vq = oracle_quantize(V.reshape(-1, d).numpy(), d, 0, w)
    shp = lambda z: {"idx": z.idx.reshape(B, Hkv, T, d), "sgn": z.sgn.reshape(B, Hkv, T, 0),
                     "norm": z.norm.reshape(B, Hkv, T), "rnorm": z.rnorm.reshape(B, Hkv, T)}
    Pi, S, c, _ = oracle_tables(d, 0, w)
    want, _ = odec.decode_attention(q.numpy(), shp(kq), shp(vq), ctx, Pi, S, c, qjl_stage=False)
    p = plan(d, 0, w)
    Kg = oracle_records_to_gpu(kq, d, 0, w)
    Vg = oracle_records_to_gpu(vq, d, 0, w, layout=vlayout)
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention(p, q.cuda(), Kg, Vg, torch.tensor(ctx, dtype=torch.int32, device="cuda"), T, Hkv,
                             out, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    assert rel_l2(out.cpu().numpy(), want) <= 1e-3


def test_search_stage1_only(gpu_lib):
    """8192 unit-norm d = 256 vectors, 16 queries, top-10, b = w = 3."""
    wl = WORKLOADS["generic"]
    d, w, k = 256, 3, 10
    X = make_generic(wl, n=8192, device="cuda")[:, :d]
    X = (X / X.norm(dim=1, keepdim=True)).contiguous()
    Q = make_generic_queries(wl, nq=16, device="cuda")[:, :d].contiguous()
    p = plan(d, 0, w)
    n = X.shape[0]
    rec = _lib.Records(n, d, 0, w)
    _lib.tq_quantize(p, X, rec)
    ws = torch.empty(_lib.tq_search_workspace_size(p, 16, n, k), dtype=torch.uint8, device="cuda")
    idx = torch.full((16, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty(16, k, device="cuda")
    _lib.tq_search_topk(p, Q, rec, n, k, idx, sc, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    got = gpu_records_to_numpy(rec, slice(0, n), d, 0, w)
    Pi, S, c, _ = oracle_tables(d, 0, w)
    osc = osearch.scores(Q.float().cpu().numpy(), got, Pi, S, c, qjl_stage=False)
    _check_topk(idx.cpu().numpy(), sc.cpu().numpy(), osc, k)
