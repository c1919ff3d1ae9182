"""Paged caches: the same decode and append through a page table.

A sequence's 256-token pages sit anywhere in the record arrays, in any order
(the online quantizer appends one vector at a time, "谷歌TurboQuant如何绕过
内存墙？" §2, so a serving cache grows by pages).  The kernels visit the same
tiles in the same order as for a contiguous cache, so the outputs must be
bit-identical to the contiguous call on the same tokens -- whose parity with
the float64 oracle the other decode tests establish -- and one case is also
checked against the oracle directly.  Pages nobody lists hold garbage.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_kv, make_queries

from parity import gpu_records_to_numpy, oracle_tables, plan, rel_l2

pytestmark = pytest.mark.gpu
BLK, ROWS = _lib.TQ_LAYOUT_BLOCK32, _lib.TQ_LAYOUT_ROWS
PAGE = 256


def _scatter(rec, units, max_pages, spare, seed, d, m, w):
    """A paged copy of a contiguous cache: pages of each unit at shuffled physical pages."""
    g = torch.Generator().manual_seed(seed)
    npages = units * max_pages + spare
    perm = torch.randperm(npages, generator=g)[:units * max_pages].to(torch.int32)
    pages = perm.reshape(units, max_pages).contiguous()
    out = _lib.Records(npages * PAGE, d, m, w, layout=rec.layout)
    fields = ("idx", "sgn", "norm", "rnorm") if m > 0 else ("idx", "norm")  # stage 1 alone: no signs
    for f in fields:
        t = getattr(out, f)
        if t.dtype == torch.int32:
            t.copy_(torch.randint(-2**31, 2**31 - 1, t.shape, generator=g, dtype=torch.int32))
        else:
            t.copy_(torch.rand(t.shape, generator=g) * 1e3)
    for u in range(units):
        for lp in range(max_pages):
            src = slice(u * max_pages * PAGE + lp * PAGE, u * max_pages * PAGE + (lp + 1) * PAGE)
            pg = int(pages[u, lp])
            dst = slice(pg * PAGE, (pg + 1) * PAGE)
            for f in fields:
                getattr(out, f)[dst] = getattr(rec, f)[src]
    return out, pages.cuda()


def _caches(B, Hkv, T, w, v_layout, seed, m=128):
    d = 128
    g = torch.Generator().manual_seed(seed)
    p = plan(d, m, w)
    K = torch.randn(B * Hkv * T, d, generator=g).cuda()
    V = torch.randn(B * Hkv * T, d, generator=g).cuda()
    Kr = _lib.Records(B * Hkv * T, d, m, w)
    Vr = _lib.Records(B * Hkv * T, d, m, w, layout=v_layout)
    _lib.tq_quantize(p, K, Kr)
    _lib.tq_quantize(p, V, Vr)
    return p, Kr, Vr


@pytest.mark.parametrize("v_layout,w,G,m", [(BLK, 2, 4, 128), (BLK, 3, 8, 128), (ROWS, 2, 4, 128), (BLK, 1, 2, 128),
                                            (BLK, 3, 4, 0), (BLK, 2, 8, 0)])
def test_paged_decode_equals_contiguous(gpu_lib, v_layout, w, G, m):
    """Tensor-core path (values in blocks) and general path (values by row); m = 0 is stage 1 alone."""
    d = 128
    B, Hkv, max_pages = 2, 3, 5
    T, Hq = max_pages * PAGE, 3 * G
    p, Kr, Vr = _caches(B, Hkv, T, w, v_layout, seed=10 * w + G, m=m)
    q = make_queries(WORKLOADS["llama8b"], B=B)[:, :Hq].float().contiguous().cuda()
    ctx = torch.tensor([T, T - 300], dtype=torch.int32, device="cuda")
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    want = torch.empty(B, Hq, d, device="cuda")
    _lib.tq_decode_attention(p, q, Kr, Vr, ctx, T, Hkv, want, ws)
    Kp, pages = _scatter(Kr, B * Hkv, max_pages, spare=4, seed=1, d=d, m=m, w=w)
    Vp, _ = _scatter(Vr, B * Hkv, max_pages, spare=4, seed=1, d=d, m=m, w=w)
    got = torch.full((B, Hq, d), float("nan"), device="cuda")
    ws.fill_(0xFF)
    _lib.tq_decode_attention_paged(p, q, Kp, Vp, ctx, pages, Hkv, got, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    assert torch.equal(got, want)


def test_paged_decode_against_oracle(gpu_lib):
    d = m = 128
    w, B, Hkv, Hq, max_pages = 2, 1, 2, 8, 3
    T = max_pages * PAGE
    p, Kr, Vr = _caches(B, Hkv, T, w, BLK, seed=3)
    Kp, pages = _scatter(Kr, B * Hkv, max_pages, spare=2, seed=2, d=d, m=m, w=w)
    Vp, _ = _scatter(Vr, B * Hkv, max_pages, spare=2, seed=2, d=d, m=m, w=w)
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(4)).cuda()
    ctx = [T - 17]
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    got = torch.empty(B, Hq, d, device="cuda")
    _lib.tq_decode_attention_paged(p, q, Kp, Vp, torch.tensor(ctx, dtype=torch.int32, device="cuda"), pages, Hkv,
                                   got, ws)
    torch.cuda.synchronize()
    rows = B * Hkv * T
    kn = gpu_records_to_numpy(Kr, slice(0, rows), d, m, w)
    vn = gpu_records_to_numpy(Vr, slice(0, rows), d, m, w)
    shape = lambda r: {"idx": r["idx"].reshape(B, Hkv, T, d), "sgn": r["sgn"].reshape(B, Hkv, T, m),
                       "norm": r["norm"].reshape(B, Hkv, T), "rnorm": r["rnorm"].reshape(B, Hkv, T)}
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.cpu().numpy(), shape(kn), shape(vn), ctx, Pi, S, c)
    assert rel_l2(got.cpu().numpy(), want) <= 1e-3


@pytest.mark.parametrize("v_layout", [BLK, ROWS])
def test_paged_append_equals_contiguous(gpu_lib, v_layout):
    """Three decode steps appended through the page table write the same words as
    the contiguous append, at the rows the table names; lengths advance alike."""
    d = m = 128
    w, B, Hkv, max_pages = 2, 2, 2, 3
    T = max_pages * PAGE
    p, Kr, Vr = _caches(B, Hkv, T, w, v_layout, seed=5)
    Kp, pages = _scatter(Kr, B * Hkv, max_pages, spare=3, seed=6, d=d, m=m, w=w)
    Vp, _ = _scatter(Vr, B * Hkv, max_pages, spare=3, seed=6, d=d, m=m, w=w)
    ctx_c = torch.tensor([255, 600], dtype=torch.int32, device="cuda")  # one append crosses a page boundary
    ctx_p = ctx_c.clone()
    g = torch.Generator().manual_seed(7)
    for _ in range(3):
        kn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
        vn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
        _lib.tq_append_kv(p, kn, vn, Kr, Vr, ctx_c, T)
        _lib.tq_append_kv_paged(p, kn, vn, Kp, Vp, ctx_p, pages)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    assert torch.equal(ctx_c, ctx_p) and ctx_c.tolist() == [258, 603]
    for u in range(B * Hkv):
        for lp in range(max_pages):
            src = slice(u * T + lp * PAGE, u * T + (lp + 1) * PAGE)
            pg = int(pages[u, lp])
            dst = slice(pg * PAGE, (pg + 1) * PAGE)
            for a, b in ((Kr, Kp), (Vr, Vp)):
                assert torch.equal(a.idx[src], b.idx[dst]) and torch.equal(a.sgn[src], b.sgn[dst])
                assert torch.equal(a.norm[src], b.norm[dst]) and torch.equal(a.rnorm[src], b.rnorm[dst])
