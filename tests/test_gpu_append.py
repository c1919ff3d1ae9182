"""GPU parity of tq_append_kv -- the new keys and values of one decode step --
against the float64 oracle.

The appended rows must follow the same rules as tq_quantize's records (index
rule, sign rule, fp32 norms; tests/parity.py); every other stored word, and
every other bit of a 32-row block word, must be left as it was; ctx_len must
advance by one except for full caches, which raise fault bit 3.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from online_kv_cache_04_b300 import _lib

from parity import (check_indices, check_norms, check_signs, gpu_records_to_numpy, oracle_quantize, oracle_tables,
                    plan, rel_l2)

pytestmark = pytest.mark.gpu
ROWS, BLK = _lib.TQ_LAYOUT_ROWS, _lib.TQ_LAYOUT_BLOCK32
FAULT_APPEND = 8


def _noise(rec, g):
    """Fill every stored word and norm with noise, so that untouched data can be checked."""
    for t in (rec.idx, rec.sgn):
        if t is not None:
            t.copy_(torch.randint(-2 ** 31, 2 ** 31 - 1, t.shape, generator=g, dtype=torch.int64).to(torch.int32))
    for t in (rec.norm, rec.rnorm):
        if t is not None:
            t.copy_(torch.rand(t.shape, generator=g) + 0.5)


def _snapshot(rec):
    return {k: (None if getattr(rec, k) is None else getattr(rec, k).cpu().clone())
            for k in ("idx", "sgn", "norm", "rnorm")}


def _check_untouched(rec, before, rows, w, d, m):
    """Rows outside `rows` keep their words and norms; block words change only at the appended rows' bits."""
    cap = rec.capacity
    keep = np.ones(cap, dtype=bool)
    keep[rows] = False
    for k in ("norm", "rnorm"):
        if before[k] is not None:
            assert torch.equal(getattr(rec, k).cpu()[torch.as_tensor(keep)], before[k][torch.as_tensor(keep)]), k
    for k, per_row in (("idx", w * d // 32), ("sgn", m // 32)):
        if before[k] is None:
            continue
        now = getattr(rec, k).cpu().numpy().view(np.uint32).reshape(-1)
        old = before[k].numpy().view(np.uint32).reshape(-1)
        if rec.layout == ROWS:
            now, old = now.reshape(cap, per_row), old.reshape(cap, per_row)
            assert np.array_equal(now[keep], old[keep]), k
        else:
            per_blk = 32 * per_row
            allowed = np.zeros(cap // 32, dtype=np.uint32)
            for r in rows:
                allowed[r // 32] |= np.uint32(1 << int((r % 32) // 2 + 16 * (r % 2)))
            diff = (now ^ old).reshape(cap // 32, per_blk)
            assert np.all((diff & ~allowed[:, None]) == 0), k


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_one_step_matches_oracle_and_leaves_the_rest(gpu_lib, w, dtype):
    d = m = 128
    B, Hkv, stride = 4, 2, 96
    ctx0 = [0, 37, 95, 96]  # empty, ragged, last free slot, full
    g = torch.Generator().manual_seed(500 + w)
    p = plan(d, m, w)
    K = _lib.Records(B * Hkv * stride, d, m, w)
    V = _lib.Records(B * Hkv * stride, d, m, w, layout=BLK)
    _noise(K, g)
    _noise(V, g)
    kb, vb = _snapshot(K), _snapshot(V)
    kn = (torch.randn(B, Hkv, d, generator=g) * (1 + 9 * (torch.rand(d, generator=g) < 0.03))).to(dtype)
    vn = torch.randn(B, Hkv, d, generator=g).to(dtype)
    kn[1, 0] = 0.0  # the zero-vector rule on the way
    ctx = torch.tensor(ctx0, dtype=torch.int32, device="cuda")
    _lib.tq_fault_flags(reset=True)
    _lib.tq_append_kv(p, kn.cuda(), vn.cuda(), K, V, ctx, stride)
    torch.cuda.synchronize()
    assert ctx.cpu().tolist() == [1, 38, 96, 96]
    assert _lib.tq_fault_flags(reset=True) == FAULT_APPEND  # the full row, and nothing else
    units = [(b, h) for b in range(B) for h in range(Hkv) if ctx0[b] < stride]
    rows = np.array([(b * Hkv + h) * stride + ctx0[b] for b, h in units])
    _, _, _, bounds = oracle_tables(d, m, w)
    for rec, new, before in ((K, kn, kb), (V, vn, vb)):
        X = np.stack([new[b, h].float().numpy() for b, h in units])
        oq = oracle_quantize(X, d, m, w)
        got = gpu_records_to_numpy(rec, rows if rec.layout == BLK else torch.as_tensor(rows, device="cuda"), d, m, w)
        ok = check_indices(got["idx"], oq, bounds)
        check_signs(got["sgn"], oq, ok, d)
        check_norms(got, oq, ok)
        _check_untouched(rec, before, rows, w, d, m)


@pytest.mark.parametrize("w", [2, 3])
def test_steps_after_a_prefill_feed_the_decode(gpu_lib, w):
    """Prefill 256 tokens per (batch row, kv head), append 3 steps, decode over all of it."""
    d = m = 128
    B, Hq, Hkv, stride = 2, 8, 2, 384
    T0 = [256, 200]
    g = torch.Generator().manual_seed(600 + w)
    p = plan(d, m, w)
    K = _lib.Records(B * Hkv * stride, d, m, w)
    V = _lib.Records(B * Hkv * stride, d, m, w, layout=BLK)
    for rec in (K, V):  # rows past the context are read by nobody, but the oracle unpacks them
        for t in (rec.idx, rec.sgn, rec.norm, rec.rnorm):
            t.zero_()
    Kx = torch.randn(B, Hkv, stride, d, generator=g).cuda()
    Vx = torch.randn(B, Hkv, stride, d, generator=g).cuda()
    for b in range(B):
        for h in range(Hkv):
            r0 = (b * Hkv + h) * stride
            _lib.tq_quantize_pair(p, Kx[b, h, :T0[b]], Vx[b, h, :T0[b]], K, V, out_offset=r0)
    ctx = torch.tensor(T0, dtype=torch.int32, device="cuda")
    for s in range(3):
        pos = [T0[b] + s for b in range(B)]
        kn = torch.stack([torch.stack([Kx[b, h, pos[b]] for h in range(Hkv)]) for b in range(B)]).contiguous()
        vn = torch.stack([torch.stack([Vx[b, h, pos[b]] for h in range(Hkv)]) for b in range(B)]).contiguous()
        _lib.tq_append_kv(p, kn, vn, K, V, ctx, stride)
    q = torch.randn(B, Hq, d, generator=g).cuda()
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, stride), dtype=torch.uint8, device="cuda")
    out = torch.empty(B, Hq, d, device="cuda")
    _lib.tq_decode_attention(p, q, K, V, ctx, stride, Hkv, out, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    assert ctx.cpu().tolist() == [T0[0] + 3, T0[1] + 3]
    # the oracle reads the records the GPU wrote (prefill and appended rows alike)
    n = B * Hkv * stride
    kr = gpu_records_to_numpy(K, slice(0, n), d, m, w)
    vr = gpu_records_to_numpy(V, slice(0, n), d, m, w)
    shp = lambda z: {k: z[k].reshape((B, Hkv, stride) + z[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.cpu().numpy(), shp(kr), shp(vr), ctx.cpu().numpy(), Pi, S, c)
    assert rel_l2(out.cpu().numpy(), want) <= 1e-3
    # the appended rows are the quantized new vectors
    units = [(b, h, T0[b] + s) for b in range(B) for h in range(Hkv) for s in range(3)]
    rows = np.array([(b * Hkv + h) * stride + t for b, h, t in units])
    X = np.stack([Kx[b, h, t].cpu().numpy() for b, h, t in units])
    oq = oracle_quantize(X, d, m, w)
    got = gpu_records_to_numpy(K, torch.as_tensor(rows, device="cuda"), d, m, w)
    _, _, _, bounds = oracle_tables(d, m, w)
    ok = check_indices(got["idx"], oq, bounds)
    check_signs(got["sgn"], oq, ok, d)
    check_norms(got, oq, ok)


def test_stage1_only_wide_vectors(gpu_lib):
    """m = 0 (no QJL rows), d = 256, w = 3, values in blocks."""
    d, m, w = 256, 0, 3
    B, Hkv, stride = 3, 2, 64
    ctx0 = [5, 63, 0]
    g = torch.Generator().manual_seed(700)
    p = plan(d, m, w)
    K = _lib.Records(B * Hkv * stride, d, m, w)
    V = _lib.Records(B * Hkv * stride, d, m, w, layout=BLK)
    _noise(K, g)
    _noise(V, g)
    kb, vb = _snapshot(K), _snapshot(V)
    kn = torch.randn(B, Hkv, d, generator=g)
    vn = torch.randn(B, Hkv, d, generator=g)
    ctx = torch.tensor(ctx0, dtype=torch.int32, device="cuda")
    _lib.tq_append_kv(p, kn.cuda(), vn.cuda(), K, V, ctx, stride)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    assert ctx.cpu().tolist() == [6, 64, 1]
    units = [(b, h) for b in range(B) for h in range(Hkv)]
    rows = np.array([(b * Hkv + h) * stride + ctx0[b] for b, h in units])
    _, _, _, bounds = oracle_tables(d, m, w)
    for rec, new, before in ((K, kn, kb), (V, vn, vb)):
        oq = oracle_quantize(np.stack([new[b, h].numpy() for b, h in units]), d, m, w)
        got = gpu_records_to_numpy(rec, rows if rec.layout == BLK else torch.as_tensor(rows, device="cuda"), d, m, w)
        ok = check_indices(got["idx"], oq, bounds)
        check_norms(got, oq, ok)
        _check_untouched(rec, before, rows, w, d, m)
