"""GPU parity of tq_decode_attention / tq_decode_scores against the float64 oracle.

Decode is compared on identical records: the oracle's own packed records fed
to the GPU (isolating decode from quantize, and checking the GPU unpacks the
oracle's words), and the GPU's records fed to the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_kv, make_queries

from parity import gpu_records_to_numpy, oracle_quantize, oracle_records_to_gpu, oracle_tables, plan, rel_l2

pytestmark = pytest.mark.gpu


def _oracle_cache_records(X, d, m, w):
    """X [B, Hkv, T, d] -> oracle Quantized (flat rows) + dict of [B, Hkv, T, ...] arrays."""
    B, H, T, _ = X.shape
    oq = oracle_quantize(X.reshape(-1, d), d, m, w)
    rec = {"idx": oq.idx.reshape(B, H, T, d), "sgn": oq.sgn.reshape(B, H, T, m),
           "norm": oq.norm.reshape(B, H, T), "rnorm": oq.rnorm.reshape(B, H, T)}
    return oq, rec


def _gpu_decode(p, q, K, V, ctx, T, Hkv, scores=False):
    B, Hq, d = q.shape
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention(p, q, K, V, ctx_t, T, Hkv, out, ws)
    sc = None
    if scores:
        sc = torch.full((B, Hq, T), float("nan"), device="cuda")
        _lib.tq_decode_scores(p, q, K, ctx_t, T, Hkv, sc, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (sc.cpu().numpy() if scores else None)


def _check(out, sc, want_out, want_sc, ctx):
    assert rel_l2(out, want_out) <= 1e-3
    if sc is not None:
        for b, L in enumerate(ctx):
            assert rel_l2(sc[b, :, :L], want_sc[b, :, :L]) <= 1e-3
            assert np.isnan(sc[b, :, L:]).all()  # untouched beyond ctx_len


@pytest.mark.parametrize("w", [1, 2, 3])
def test_tiny_workload_oracle_records(gpu_lib, w):
    wl = WORKLOADS["tiny"]
    d = m = 128
    K = make_kv(wl, which=0).numpy()
    V = make_kv(wl, which=1).numpy()
    q = make_queries(wl)
    T = K.shape[2]
    Pi, S, c, _ = oracle_tables(d, m, w)
    kq, krec = _oracle_cache_records(K, d, m, w)
    vq, vrec = _oracle_cache_records(V, d, m, w)
    want_out, want_sc = odec.decode_attention(q.numpy(), krec, vrec, [T], Pi, S, c)
    p = plan(d, m, w)
    out, sc = _gpu_decode(p, q.cuda(), oracle_records_to_gpu(kq, d, m, w), oracle_records_to_gpu(vq, d, m, w),
                          [T], T, 1, scores=True)
    _check(out, sc, want_out, want_sc, [T])


@pytest.mark.parametrize("w", [1, 2, 3])
def test_gqa_ragged_batch_gpu_records(gpu_lib, w):
    """B = 3 rows with ctx 700, 1, 0 of capacity 700; 16 / 4 heads; bf16 queries and cache."""
    wl = WORKLOADS["llama8b"]
    d = m = 128
    B, Hq, Hkv, T = 3, 16, 4, 700
    K = make_kv(wl, B=B, T=T, which=0)[:, :Hkv]
    V = make_kv(wl, B=B, T=T, which=1)[:, :Hkv]
    q = make_queries(wl, B=B)[:, :Hq]
    ctx = [700, 1, 0]
    p = plan(d, m, w)
    Kr = _lib.Records(B * Hkv * T, d, m, w)
    Vr = _lib.Records(B * Hkv * T, d, m, w)
    _lib.tq_quantize(p, K.reshape(-1, d).cuda(), Kr)
    _lib.tq_quantize(p, V.reshape(-1, d).cuda(), Vr)
    out, sc = _gpu_decode(p, q.contiguous().cuda(), Kr, Vr, ctx, T, Hkv, scores=True)
    # oracle on the GPU's own records
    rows = slice(0, B * Hkv * T)
    kg = gpu_records_to_numpy(Kr, rows, d, m, w)
    vg = gpu_records_to_numpy(Vr, rows, d, m, w)
    shp = lambda r: {k: r[k].reshape((B, Hkv, T) + r[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
    Pi, S, c, _ = oracle_tables(d, m, w)
    want_out, want_sc = odec.decode_attention(q.float().numpy(), shp(kg), shp(vg), ctx, Pi, S, c)
    _check(out, sc, want_out, want_sc, ctx)
    assert np.all(out[2] == 0.0)  # ctx_len 0 -> zeros


def test_context_length_one_and_explicit_scale(gpu_lib):
    d = m = 128
    w = 2
    g = torch.Generator().manual_seed(0)
    K = torch.randn(1, 2, 50, d, generator=g)
    V = torch.randn(1, 2, 50, d, generator=g)
    q = torch.randn(1, 4, d, generator=g)
    p = plan(d, m, w)
    kq, krec = _oracle_cache_records(K.numpy(), d, m, w)
    vq, vrec = _oracle_cache_records(V.numpy(), d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    B, Hq, Hkv, T = 1, 4, 2, 50
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    out = torch.empty(B, Hq, d, device="cuda")
    for L, scale in ((1, 0.0), (50, 0.3)):
        ctx_t = torch.tensor([L], dtype=torch.int32, device="cuda")
        _lib.tq_decode_attention(p, q.cuda(), oracle_records_to_gpu(kq, d, m, w), oracle_records_to_gpu(vq, d, m, w),
                                 ctx_t, T, Hkv, out, ws, scale=scale)
        want, _ = odec.decode_attention(q.numpy(), krec, vrec, [L], Pi, S, c, scale=scale or None)
        assert rel_l2(out.cpu().numpy(), want) <= 1e-3


def test_llama8b_full_size(gpu_lib):
    """32 / 8 heads, d = 128, ctx 32768, b = 3 and 4: GPU quantize + decode; oracle decode on the GPU records."""
    wl = WORKLOADS["llama8b"]
    d = m = 128
    B, Hq, Hkv, T = 1, 32, 8, 32768
    K = make_kv(wl, which=0, device="cuda")
    V = make_kv(wl, which=1, device="cuda")
    q = make_queries(wl, device="cuda")
    for w in (2, 3):
        p = plan(d, m, w)
        Kr = _lib.Records(B * Hkv * T, d, m, w)
        Vr = _lib.Records(B * Hkv * T, d, m, w)
        _lib.tq_quantize(p, K.reshape(-1, d), Kr)
        _lib.tq_quantize(p, V.reshape(-1, d), Vr)
        out, sc = _gpu_decode(p, q, Kr, Vr, [T], T, Hkv, scores=True)
        rows = slice(0, B * Hkv * T)
        kg = gpu_records_to_numpy(Kr, rows, d, m, w)
        vg = gpu_records_to_numpy(Vr, rows, d, m, w)
        shp = lambda r: {k: r[k].reshape((B, Hkv, T) + r[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
        Pi, S, c, _ = oracle_tables(d, m, w)
        want_out, want_sc = odec.decode_attention(q.float().cpu().numpy(), shp(kg), shp(vg), [T], Pi, S, c)
        _check(out, sc, want_out, want_sc, [T])


@pytest.mark.parametrize("w", [2])
def test_longctx_full_size_sampled(gpu_lib, w):
    """Batch 16, ctx 131072, 8 kv heads: full GPU path; oracle on (b, h) = (0, 0), (15, 7)."""
    wl = WORKLOADS["longctx"]
    d = m = 128
    B, Hq, Hkv, T = 16, 32, 8, 131072
    p = plan(d, m, w)
    q = make_queries(wl, device="cuda")
    Kr = _lib.Records(B * Hkv * T, d, m, w)
    Vr = _lib.Records(B * Hkv * T, d, m, w)
    for which, rec in ((0, Kr), (1, Vr)):
        for b0 in range(0, B, 4):  # generate in slices to bound memory
            X = make_kv(wl, B=4, which=which, device="cuda")
            _lib.tq_quantize(p, X.reshape(-1, d), rec, out_offset=b0 * Hkv * T)
            del X
    ctx = [T - 37 * b for b in range(B)]
    out, _ = _gpu_decode(p, q, Kr, Vr, ctx, T, Hkv)
    Pi, S, c, _ = oracle_tables(d, m, w)
    for b, h in ((0, 0), (15, 7)):
        rows = slice((b * Hkv + h) * T, (b * Hkv + h + 1) * T)
        kg = gpu_records_to_numpy(Kr, rows, d, m, w)
        vg = gpu_records_to_numpy(Vr, rows, d, m, w)
        shp = lambda r: {k: r[k].reshape((1, 1, T) + r[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
        qs = q[b:b + 1, h * 4:(h + 1) * 4].float().cpu().numpy()
        want, _ = odec.decode_attention(qs, shp(kg), shp(vg), [ctx[b]], Pi, S, c)
        assert rel_l2(out[b, h * 4:(h + 1) * 4], want[0]) <= 1e-3


@pytest.mark.parametrize("w", [1, 2, 3])
def test_block_layout_values_oracle_records(gpu_lib, w):
    """V records in 32-row blocks (any shape takes the general kernel): oracle-packed, ragged lengths."""
    d = m = 128
    g = torch.Generator().manual_seed(40 + w)
    B, Hq, Hkv, T = 2, 6, 2, 96
    K = torch.randn(B, Hkv, T, d, generator=g)
    V = torch.randn(B, Hkv, T, d, generator=g) * 3
    q = torch.randn(B, Hq, d, generator=g)
    kq, krec = _oracle_cache_records(K.numpy(), d, m, w)
    vq, vrec = _oracle_cache_records(V.numpy(), d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    ctx = [96, 45]
    want, _ = odec.decode_attention(q.numpy(), krec, vrec, ctx, Pi, S, c)
    p = plan(d, m, w)
    Kr = oracle_records_to_gpu(kq, d, m, w)
    Vr = oracle_records_to_gpu(vq, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    out, _ = _gpu_decode(p, q.cuda(), Kr, Vr, ctx, T, Hkv)
    assert rel_l2(out, want) <= 1e-3
