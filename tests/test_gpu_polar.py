"""GPU parity of the PolarQuant stage (+ QJL) against the float64 oracle.

Codes: at least 99.99 % of angle codes equal per level; every mismatch is an
adjacent cell (cyclically at level 1) with the oracle's angle within 1e-5 of
the boundary between them (the fp32 rotation and atan2 against float64).
Norms within 4e-7 relative; residual norms (1e-4) and signs (the rule of
tests/parity.py) on vectors whose codes all match.  Decode: relative L2 <=
1e-3 on the oracle's records and on the GPU's own records.
"""

import numpy as np
import pytest
import torch

from oracle import polar
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import POLAR_SEEDS, WORKLOADS, make_kv

from parity import rel_l2

pytestmark = pytest.mark.gpu
_CACHE = {}


def _tables(d):
    if d not in _CACHE:
        rs, qs = POLAR_SEEDS
        plan = _lib.PolarPlan(d, d, 4, 2, rs, qs)
        cb = polar.PolarCodebooks(d=d, b1=4, b=2, books=[(np.asarray(c), np.asarray(b)) for c, b in plan.books])
        _CACHE[d] = (plan, cb, plan.pi, plan.S)
    return _CACHE[d]


def _check_codes(got, want_angles, cb):
    all_ok = np.ones(got[0].shape[0], dtype=bool)
    for lev, (g, ang, (c, bd)) in enumerate(zip(got, want_angles, cb.books), start=1):
        w = np.searchsorted(bd, ang, side="left")
        eq = g == w
        assert eq.mean() >= 0.9999, (lev, eq.mean())
        n = len(c)
        for v, i in np.argwhere(~eq):
            a, b = int(g[v, i]), int(w[v, i])
            diff = (a - b) % n if lev == 1 else abs(a - b)
            assert diff in (1, n - 1) if lev == 1 else diff == 1, (lev, a, b)
            edges = np.concatenate([bd, [0.0, 2 * np.pi]]) if lev == 1 else bd
            assert np.min(np.abs(edges - ang[v, i])) <= 1e-5, (lev, ang[v, i])
        all_ok &= eq.all(axis=1)
    return all_ok


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [128, 64])
def test_quantize_polar_matches_oracle(gpu_lib, dtype, d):
    plan, cb, Pi, S = _tables(d)
    wl = WORKLOADS["llama8b"]
    X = make_kv(wl, B=1, T=2500, which=1)[0, 2, :, :d].to(dtype)
    n = X.shape[0]
    rec = plan.records(n + 3)
    _lib.tq_quantize_polar(plan, X.cuda(), rec, out_offset=3)
    torch.cuda.synchronize()
    oq = polar.quantize_polar(X.float().numpy(), Pi, S, cb)
    words = rec.idx[3:].cpu().numpy().view(np.uint32)
    got = polar.unpack_indices(words, d)
    ok = _check_codes(got, oq.angles, cb)
    assert ok.mean() > 0.99
    # the packed words are exactly the oracle packer's image of the codes
    assert np.array_equal(words, polar.pack_indices(got, d))
    n64 = oq.norm.astype(np.float64)
    assert np.all(np.abs(rec.norm[3:].cpu().numpy() - n64) <= 4e-7 * n64)
    rn = rec.rnorm[3:].cpu().numpy()[ok]
    r64 = oq.rnorm.astype(np.float64)[ok]
    assert np.all(np.abs(rn - r64) <= 1e-4 * r64 + 1e-6 * n64[ok])
    sg = np.unpackbits(rec.sgn[3:].cpu().numpy().view(np.uint8), bitorder="little").reshape(n, d).astype(bool)
    eq = sg[ok] == oq.sgn[ok]
    assert eq.mean() >= 0.9999


def _polar_case(d, B, Hq, Hkv, T, ctx, seed, own, q_dtype=torch.float32):
    plan, cb, Pi, S = _tables(d)
    wl = WORKLOADS["llama8b"]
    K = make_kv(wl, B=B, T=T, which=0)[:, :Hkv, :, :d].float().reshape(-1, d)
    V = make_kv(wl, B=B, T=T, which=1)[:, :Hkv, :, :d].float().reshape(-1, d)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g).to(q_dtype)
    rows = K.shape[0]
    if own:
        Kr, Vr = plan.records(rows), plan.records(rows)
        _lib.tq_quantize_polar(plan, K.cuda(), Kr)
        _lib.tq_quantize_polar(plan, V.cuda(), Vr)
        torch.cuda.synchronize()

        def back(r):
            idx = polar.unpack_indices(r.idx.cpu().numpy().view(np.uint32), d)
            sgn = np.unpackbits(r.sgn.cpu().numpy().view(np.uint8), bitorder="little").reshape(rows, d).astype(bool)
            return polar.PolarQuantized(idx=idx, norm=r.norm.cpu().numpy(), sgn=sgn, rnorm=r.rnorm.cpu().numpy(),
                                        angles=None)
        oK, oV = back(Kr), back(Vr)
    else:
        oK = polar.quantize_polar(K.numpy(), Pi, S, cb)
        oV = polar.quantize_polar(V.numpy(), Pi, S, cb)

        def up(o):
            t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
            return _lib.Records.wrap(t(polar.pack_indices(o.idx, d).view(np.int32)),
                                     t(np.packbits(o.sgn, axis=1, bitorder="little").view(np.int32)), t(o.norm),
                                     t(o.rnorm), d, d, 0)
        Kr, Vr = up(oK), up(oV)
    want, _ = polar.decode_attention_polar(q.float().numpy(), oK, oV, (B, Hkv, T), ctx, Pi, S, cb)
    ws = torch.empty(_lib.tq_decode_polar_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention_polar(plan, q.cuda(), Kr, Vr, torch.tensor(ctx, dtype=torch.int32, device="cuda"), T,
                                   Hkv, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), want


@pytest.mark.parametrize("d", [128, 64])
def test_decode_polar_on_oracle_records(gpu_lib, d):
    out, want = _polar_case(d, 2, 8, 2, 777, [777, 300], 41, own=False)
    assert rel_l2(out, want) <= 1e-3


def test_decode_polar_on_gpu_records_bf16_query(gpu_lib):
    out, want = _polar_case(128, 1, 4, 1, 2048, [2048], 43, own=True, q_dtype=torch.bfloat16)
    assert rel_l2(out, want) <= 1e-3


def test_decode_polar_single_token_and_empty_row(gpu_lib):
    out, want = _polar_case(128, 2, 8, 1, 256, [1, 0], 45, own=False)
    assert rel_l2(out[:1], want[:1]) <= 1e-3
    assert np.all(out[1] == 0.0)
