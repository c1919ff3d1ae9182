"""GPU parity of the tensor-core decode path (values in 32-row blocks, d = m = 128).

tq_decode_attention takes the warp-MMA (mma.sync f16) kernel when the value
records are in TQ_LAYOUT_BLOCK32, ctx_stride is a multiple of 128 and there are at most 8
query heads per kv head.  Outputs are compared with the float64 oracle on
identical records (the oracle's own packed records, or the GPU's records
unpacked by the oracle), relative L2 <= 1e-3.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_kv, make_queries

from parity import gpu_records_to_numpy, oracle_quantize, oracle_records_to_gpu, oracle_tables, plan, rel_l2

pytestmark = pytest.mark.gpu
BLK = _lib.TQ_LAYOUT_BLOCK32


def _oracle_recs(X, d, m, w):
    B, H, T, _ = X.shape
    oq = oracle_quantize(X.reshape(-1, d), d, m, w)
    rec = {"idx": oq.idx.reshape(B, H, T, d), "sgn": oq.sgn.reshape(B, H, T, m),
           "norm": oq.norm.reshape(B, H, T), "rnorm": oq.rnorm.reshape(B, H, T)}
    return oq, rec


def _decode(p, q, K, V, ctx, T, Hkv):
    B, Hq, d = q.shape
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # stale NaN patterns must never be read
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention(p, q, K, V, ctx_t, T, Hkv, out, ws)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    return out.cpu().numpy()


def _case(B, Hq, Hkv, T, ctx, w, seed, kscale=None, vscale=None):
    d = m = 128
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    V = torch.randn(B, Hkv, T, d, generator=g)
    if kscale is not None:
        K = K * kscale(T)[None, None, :, None]
    if vscale is not None:
        V = V * vscale(T)[None, None, :, None]
    q = torch.randn(B, Hq, d, generator=g)
    kq, krec = _oracle_recs(K.numpy(), d, m, w)
    vq, vrec = _oracle_recs(V.numpy(), d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.numpy(), krec, vrec, ctx, Pi, S, c)
    p = plan(d, m, w)
    out = _decode(p, q.cuda(), oracle_records_to_gpu(kq, d, m, w), oracle_records_to_gpu(vq, d, m, w, layout=BLK),
                  ctx, T, Hkv)
    return out, want


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (8, 1), (3, 3), (6, 2)])
def test_oracle_records_gqa_shapes(gpu_lib, w, Hq, Hkv):
    out, want = _case(2, Hq, Hkv, 640, [640, 333], w, seed=10 * w + Hq)
    assert rel_l2(out, want) <= 1e-3


def test_units_split_across_ctas_ragged_and_empty(gpu_lib):
    """4 x 4 units of 20 tiles over at most 148 CTAs: CTAs span unit boundaries; ctx 0 and 1 rows."""
    B, Hq, Hkv, T = 4, 16, 4, 2560
    out, want = _case(B, Hq, Hkv, T, [2560, 1999, 1, 0], 2, seed=3)
    assert rel_l2(out[:3], want[:3]) <= 1e-3
    assert np.all(out[3] == 0.0)


def test_lazy_rescale_and_value_norm_range(gpu_lib):
    """Later keys score far higher (forces the running reference up) and value norms span 1e-3..1e3."""
    ks = lambda T: torch.where(torch.arange(T) >= 700, 6.0, 1.0)
    vs = lambda T: torch.exp(torch.linspace(-7.0, 7.0, T))
    out, want = _case(1, 8, 2, 1408, [1408], 2, seed=5, kscale=ks, vscale=vs)
    assert rel_l2(out, want) <= 1e-3


@pytest.mark.parametrize("w", [1, 2, 3])
def test_rescale_within_a_cta(gpu_lib, w):
    """512 tiles of one kv head over at most 148 CTAs (several tiles each); key scale cycles
    1, 2, 4, 8 per tile so the running reference jumps inside a CTA's range."""
    ks = lambda T: 2.0 ** ((torch.arange(T) // 128) % 4).float()
    vs = lambda T: torch.exp(torch.sin(torch.arange(T).float() / 300.0) * 4.0)
    out, want = _case(1, 4, 1, 65536, [65536], w, seed=17 + w, kscale=ks, vscale=vs)
    assert rel_l2(out, want) <= 1e-3


@pytest.mark.parametrize("w", [2, 3])
def test_llama8b_full_size_gpu_records(gpu_lib, w):
    """32 / 8 heads, ctx 32768, bf16 K/V: GPU quantize (keys by row, values in blocks), tensor-core decode."""
    wl = WORKLOADS["llama8b"]
    d = m = 128
    B, Hq, Hkv, T = 1, 32, 8, 32768
    K = make_kv(wl, which=0, device="cuda")
    V = make_kv(wl, which=1, device="cuda")
    q = make_queries(wl, device="cuda")
    p = plan(d, m, w)
    Kr = _lib.Records(B * Hkv * T, d, m, w)
    Vr = _lib.Records(B * Hkv * T, d, m, w, layout=BLK)
    _lib.tq_quantize(p, K.reshape(-1, d), Kr)
    _lib.tq_quantize(p, V.reshape(-1, d), Vr)
    out = _decode(p, q, Kr, Vr, [T], T, Hkv)
    rows = slice(0, B * Hkv * T)
    kg = gpu_records_to_numpy(Kr, rows, d, m, w)
    vg = gpu_records_to_numpy(Vr, rows, d, m, w)
    shp = lambda r: {k: r[k].reshape((B, Hkv, T) + r[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.float().cpu().numpy(), shp(kg), shp(vg), [T], Pi, S, c)
    assert rel_l2(out, want) <= 1e-3


@pytest.mark.parametrize("w", [1, 2, 3])
def test_longctx_full_size_sampled(gpu_lib, w):
    """Batch 16, ctx 131072, 8 kv heads (GQA 4:1), b = w + 1; oracle on (b, h) = (0, 0), (9, 3), (15, 7)."""
    wl = WORKLOADS["longctx"]
    d = m = 128
    B, Hq, Hkv, T = 16, 32, 8, 131072
    p = plan(d, m, w)
    q = make_queries(wl, device="cuda")
    Kr = _lib.Records(B * Hkv * T, d, m, w)
    Vr = _lib.Records(B * Hkv * T, d, m, w, layout=BLK)
    for which, rec in ((0, Kr), (1, Vr)):
        for b0 in range(0, B, 4):  # generate in slices to bound memory
            X = make_kv(wl, B=4, which=which, device="cuda")
            _lib.tq_quantize(p, X.reshape(-1, d), rec, out_offset=b0 * Hkv * T)
            del X
    ctx = [T - 37 * b for b in range(B)]
    out = _decode(p, q, Kr, Vr, ctx, T, Hkv)
    Pi, S, c, _ = oracle_tables(d, m, w)
    for b, h in ((0, 0), (9, 3), (15, 7)):
        rows = slice((b * Hkv + h) * T, (b * Hkv + h + 1) * T)
        kg = gpu_records_to_numpy(Kr, rows, d, m, w)
        vg = gpu_records_to_numpy(Vr, rows, d, m, w)
        shp = lambda r: {k: r[k].reshape((1, 1, T) + r[k].shape[1:]) for k in ("idx", "sgn", "norm", "rnorm")}
        qs = q[b:b + 1, h * 4:(h + 1) * 4].float().cpu().numpy()
        want, _ = odec.decode_attention(qs, shp(kg), shp(vg), [ctx[b]], Pi, S, c)
        assert rel_l2(out[b, h * 4:(h + 1) * 4], want[0]) <= 1e-3


def test_tiny_workload_g8(gpu_lib):
    """One kv head, 8 query heads, 4096 fp32 keys/values with outlier channels, b = 3."""
    wl = WORKLOADS["tiny"]
    d = m = 128
    w = 2
    K = make_kv(wl, which=0).numpy()
    V = make_kv(wl, which=1).numpy()
    q = make_queries(wl)
    T = K.shape[2]
    kq, krec = _oracle_recs(K, d, m, w)
    vq, vrec = _oracle_recs(V, d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.numpy(), krec, vrec, [T], Pi, S, c)
    out = _decode(plan(d, m, w), q.cuda(), oracle_records_to_gpu(kq, d, m, w),
                  oracle_records_to_gpu(vq, d, m, w, layout=BLK), [T], T, 1)
    assert rel_l2(out, want) <= 1e-3


@pytest.mark.parametrize("G", [4, 8])
def test_one_unit_over_all_ctas_repeated_calls(gpu_lib, G):
    """One kv head with G query heads and 512 tiles of 128 tokens: every CTA of the grid (three
    per SM at 4 heads, two at 8) holds a part of the one unit, the most partials a unit can have.
    Decoded three times through one workspace: each call gives the same result (up to the order
    of the in-block float atomics of the query offsets)."""
    d = m = 128
    w = 2
    T = 65536
    g = torch.Generator().manual_seed(29)
    K = torch.randn(1, 1, T, d, generator=g)
    V = torch.randn(1, 1, T, d, generator=g)
    q = torch.randn(1, G, d, generator=g)
    kq, krec = _oracle_recs(K.numpy(), d, m, w)
    vq, vrec = _oracle_recs(V.numpy(), d, m, w)
    Pi, S, c, _ = oracle_tables(d, m, w)
    want, _ = odec.decode_attention(q.numpy(), krec, vrec, [T - 5], Pi, S, c)
    p = plan(d, m, w)
    Kg = oracle_records_to_gpu(kq, d, m, w)
    Vg = oracle_records_to_gpu(vq, d, m, w, layout=BLK)
    ws = torch.empty(_lib.tq_decode_workspace_size(p, 1, G, 1, T), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    ctx_t = torch.tensor([T - 5], dtype=torch.int32, device="cuda")
    qd = q.cuda()
    outs = []
    for _ in range(3):
        out = torch.full((1, G, d), float("nan"), device="cuda")
        _lib.tq_decode_attention(p, qd, Kg, Vg, ctx_t, T, 1, out, ws)
        torch.cuda.synchronize()
        assert _lib.tq_fault_flags() == 0
        outs.append(out.cpu().numpy())
    assert rel_l2(outs[0], want) <= 1e-3
    assert rel_l2(outs[1], outs[0]) <= 1e-6 and rel_l2(outs[2], outs[0]) <= 1e-6
