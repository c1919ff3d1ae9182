"""GPU parity of tq_decode_attention_append -- a decode step with the online
append fused in -- against the float64 oracle.

The appended rows follow tq_quantize's rules (index, sign and norm rules of
tests/parity.py); every other stored word and block bit is left as it was;
ctx_len advances by one except for full caches (fault bit 3); the attention
output is the oracle's decode over the records the GPU holds after the step,
with the advanced lengths ("谷歌TurboQuant如何绕过内存墙？" §2: the quantizer
runs per vector as tokens arrive).  Paged caches give bit-identical results to
contiguous ones, and the fused step agrees with tq_append_kv followed by
tq_decode_attention.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from online_kv_cache_04_b300 import _lib

from parity import (check_indices, check_norms, check_signs, gpu_records_to_numpy, oracle_quantize, oracle_tables,
                    plan, rel_l2)
from test_gpu_append import _check_untouched, _noise, _snapshot

pytestmark = pytest.mark.gpu
ROWS, BLK = _lib.TQ_LAYOUT_ROWS, _lib.TQ_LAYOUT_BLOCK32
FAULT_APPEND = 8
PAGE = 256


def _oracle_decode(q, K, V, ctx, B, Hkv, stride, d, m, w):
    n = B * Hkv * stride
    kr = gpu_records_to_numpy(K, slice(0, n), d, m, w)
    vr = gpu_records_to_numpy(V, slice(0, n), d, m, w)
    shp = lambda z: {k: z[k].reshape((B, Hkv, stride) + z[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.cpu().numpy(), shp(kr), shp(vr), np.asarray(ctx), Pi, S, c,
                                    qjl_stage=m > 0)
    return want


def _workspace(p, B, Hq, Hkv, stride):
    return torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, stride), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("w,m", [(1, 128), (2, 128), (3, 128), (2, 0)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("v_layout", [BLK, ROWS])
def test_fused_step_matches_oracle_and_leaves_the_rest(gpu_lib, w, m, dtype, v_layout):
    """Values in blocks take the tensor-core launches (append inside them); values by
    row the general path (tq_append_kv's launches first).  Rows: empty, ragged,
    last free slot, full."""
    d = 128
    B, Hq, Hkv, stride = 4, 8, 2, 512
    ctx0 = [0, 37, 511, 512]
    g = torch.Generator().manual_seed(900 + 10 * w + m + (dtype == torch.bfloat16) + 3 * v_layout)
    p = plan(d, m, w)
    K = _lib.Records(B * Hkv * stride, d, m, w)
    V = _lib.Records(B * Hkv * stride, d, m, w, layout=v_layout)
    _noise(K, g)
    _noise(V, g)
    kb, vb = _snapshot(K), _snapshot(V)
    kn = (torch.randn(B, Hkv, d, generator=g) * (1 + 9 * (torch.rand(d, generator=g) < 0.03))).to(dtype)
    vn = torch.randn(B, Hkv, d, generator=g).to(dtype)
    kn[1, 0] = 0.0  # the zero-vector rule on the way
    q = torch.randn(B, Hq, d, generator=g).cuda()
    ctx = torch.tensor(ctx0, dtype=torch.int32, device="cuda")
    ws = _workspace(p, B, Hq, Hkv, stride)
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_fault_flags(reset=True)
    _lib.tq_decode_attention_append(p, q, kn.cuda(), vn.cuda(), K, V, ctx, stride, Hkv, out, ws)
    torch.cuda.synchronize()
    assert ctx.cpu().tolist() == [1, 38, 512, 512]
    assert _lib.tq_fault_flags(reset=True) == FAULT_APPEND  # the full row, and nothing else
    units = [(b, h) for b in range(B) for h in range(Hkv) if ctx0[b] < stride]
    rows = np.array([(b * Hkv + h) * stride + ctx0[b] for b, h in units])
    _, _, _, bounds = oracle_tables(d, m, w)
    for rec, new, before in ((K, kn, kb), (V, vn, vb)):
        X = np.stack([new[b, h].float().numpy() for b, h in units])
        oq = oracle_quantize(X, d, m, w)
        got = gpu_records_to_numpy(rec, rows if rec.layout == BLK else torch.as_tensor(rows, device="cuda"), d, m, w)
        ok = check_indices(got["idx"], oq, bounds)
        if m > 0:
            check_signs(got["sgn"], oq, ok, d)
        check_norms(got, oq, ok)
        _check_untouched(rec, before, rows, w, d, m)
    want = _oracle_decode(q, K, V, ctx.cpu().tolist(), B, Hkv, stride, d, m, w)
    assert rel_l2(out.cpu().numpy(), want) <= 1e-3


@pytest.mark.parametrize("w", [2, 3])
def test_fused_steps_agree_with_append_then_decode(gpu_lib, w):
    """Prefill, then four steps crossing a 256-token tile boundary, fused on one copy of
    the caches and as tq_append_kv + tq_decode_attention on another."""
    d = m = 128
    B, Hq, Hkv, stride = 2, 16, 2, 1024
    T0 = [254, 700]
    g = torch.Generator().manual_seed(950 + w)
    p = plan(d, m, w)
    caches = []
    for _ in range(2):
        K = _lib.Records(B * Hkv * stride, d, m, w)
        V = _lib.Records(B * Hkv * stride, d, m, w, layout=BLK)
        for rec in (K, V):
            for t in (rec.idx, rec.sgn, rec.norm, rec.rnorm):
                t.zero_()
        caches.append((K, V))
    Kx = torch.randn(B, Hkv, stride, d, generator=g).to(torch.bfloat16).cuda()
    Vx = torch.randn(B, Hkv, stride, d, generator=g).to(torch.bfloat16).cuda()
    for K, V in caches:
        for b in range(B):
            for h in range(Hkv):
                r0 = (b * Hkv + h) * stride
                _lib.tq_quantize_pair(p, Kx[b, h, :T0[b]], Vx[b, h, :T0[b]], K, V, out_offset=r0)
    ctx_f = torch.tensor(T0, dtype=torch.int32, device="cuda")
    ctx_s = ctx_f.clone()
    ws = _workspace(p, B, Hq, Hkv, stride)
    for s in range(4):
        pos = [T0[b] + s for b in range(B)]
        kn = torch.stack([torch.stack([Kx[b, h, pos[b]] for h in range(Hkv)]) for b in range(B)]).contiguous()
        vn = torch.stack([torch.stack([Vx[b, h, pos[b]] for h in range(Hkv)]) for b in range(B)]).contiguous()
        q = torch.randn(B, Hq, d, generator=g).cuda()
        of = torch.empty(B, Hq, d, device="cuda")
        os_ = torch.empty(B, Hq, d, device="cuda")
        (Kf, Vf), (Ks, Vs) = caches
        _lib.tq_decode_attention_append(p, q, kn, vn, Kf, Vf, ctx_f, stride, Hkv, of, ws)
        _lib.tq_append_kv(p, kn, vn, Ks, Vs, ctx_s, stride)
        _lib.tq_decode_attention(p, q, Ks, Vs, ctx_s, stride, Hkv, os_, ws)
        torch.cuda.synchronize()
        assert _lib.tq_fault_flags() == 0
        assert ctx_f.cpu().tolist() == ctx_s.cpu().tolist() == [T0[b] + s + 1 for b in range(B)]
        assert rel_l2(of.cpu().numpy(), os_.cpu().numpy()) <= 1e-3
        want = _oracle_decode(q, Kf, Vf, ctx_f.cpu().tolist(), B, Hkv, stride, d, m, w)
        assert rel_l2(of.cpu().numpy(), want) <= 1e-3
    # the appended rows of the fused copy are the quantized new vectors
    Kf, _ = caches[0]
    units = [(b, h, T0[b] + s) for b in range(B) for h in range(Hkv) for s in range(4)]
    rows = np.array([(b * Hkv + h) * stride + t for b, h, t in units])
    oq = oracle_quantize(np.stack([Kx[b, h, t].float().cpu().numpy() for b, h, t in units]), d, m, w)
    got = gpu_records_to_numpy(Kf, torch.as_tensor(rows, device="cuda"), d, m, w)
    _, _, _, bounds = oracle_tables(d, m, w)
    ok = check_indices(got["idx"], oq, bounds)
    check_signs(got["sgn"], oq, ok, d)
    check_norms(got, oq, ok)


def test_fused_paged_equals_contiguous(gpu_lib):
    """The same step through a page table: the same records at the rows the table
    names and bit-identical outputs; one append lands on a fresh page."""
    d = m = 128
    w, B, Hq, Hkv, max_pages = 2, 2, 8, 2, 3
    stride = max_pages * PAGE
    g = torch.Generator().manual_seed(990)
    p = plan(d, m, w)
    K = _lib.Records(B * Hkv * stride, d, m, w)
    V = _lib.Records(B * Hkv * stride, d, m, w, layout=BLK)
    X = torch.randn(2, B * Hkv * stride, d, generator=g).cuda()
    _lib.tq_quantize(p, X[0], K)
    _lib.tq_quantize(p, X[1], V)
    units = B * Hkv
    npages = units * max_pages + 2
    pages = torch.randperm(npages, generator=g)[:units * max_pages].to(torch.int32).reshape(units, max_pages)
    Kp = _lib.Records(npages * PAGE, d, m, w)
    Vp = _lib.Records(npages * PAGE, d, m, w, layout=BLK)
    for src, dst in ((K, Kp), (V, Vp)):
        for f in ("idx", "sgn", "norm", "rnorm"):
            t = getattr(dst, f)
            t.zero_()
            for u in range(units):
                for lp in range(max_pages):
                    pg = int(pages[u, lp])
                    t[pg * PAGE:(pg + 1) * PAGE] = getattr(src, f)[u * stride + lp * PAGE:u * stride + (lp + 1) * PAGE]
    pages = pages.cuda()
    ctx_c = torch.tensor([256, 401], dtype=torch.int32, device="cuda")  # row 0 appends on its second page
    ctx_p = ctx_c.clone()
    ws = _workspace(p, B, Hq, Hkv, stride)
    q = torch.randn(B, Hq, d, generator=g).cuda()
    kn = torch.randn(B, Hkv, d, generator=g).cuda()
    vn = torch.randn(B, Hkv, d, generator=g).cuda()
    oc = torch.empty(B, Hq, d, device="cuda")
    op = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention_append(p, q, kn, vn, K, V, ctx_c, stride, Hkv, oc, ws)
    _lib.tq_decode_attention_append(p, q, kn, vn, Kp, Vp, ctx_p, stride, Hkv, op, ws, pages=pages)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    assert ctx_c.cpu().tolist() == ctx_p.cpu().tolist() == [257, 402]
    assert torch.equal(oc, op)
    for u in range(units):
        for lp in range(max_pages):
            pg = int(pages[u, lp])
            for a, b in ((K, Kp), (V, Vp)):
                for f in ("idx", "sgn", "norm", "rnorm"):
                    assert torch.equal(getattr(a, f)[u * stride + lp * PAGE:u * stride + (lp + 1) * PAGE],
                                       getattr(b, f)[pg * PAGE:(pg + 1) * PAGE])
