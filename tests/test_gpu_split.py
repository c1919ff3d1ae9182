"""GPU parity of outlier-channel split precision against the float64 oracle.

The channels of a head split into outliers (b + 1 total bits) and the rest
(b bits), each side its own instance ("TurboQuant压缩效果": the 2.5 / 3.5-bit
settings); here d = 128 with half the channels promoted, the split those
labels need.  Quantize: the index, sign and norm rules of tests/parity.py on
each side.  Decode: relative L2 <= 1e-3 on the oracle's records and on the
GPU's own records.
"""

import numpy as np
import pytest
import torch

from oracle import mixed
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import SPLIT_SEEDS, WORKLOADS, make_kv, make_queries

from parity import check_indices, check_norms, check_signs, gpu_records_to_numpy, oracle_records_to_gpu, rel_l2

pytestmark = pytest.mark.gpu
D, NO = 128, 64


def _setup(bits, X_sample):
    perm = mixed.choose_outliers(X_sample, NO)
    (ro, qo), (rr, qr) = SPLIT_SEEDS["outlier"], SPLIT_SEEDS["regular"]
    t = mixed.make_tables(perm, NO, bits, ro, qo, rr, qr)
    po = _lib.Plan(NO, NO, bits, ro, qo)
    pr = _lib.Plan(D - NO, D - NO, bits - 1, rr, qr)
    perm_d = torch.from_numpy(perm.astype(np.int32)).cuda()
    return t, po, pr, perm_d


@pytest.mark.parametrize("bits", [2, 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_split_matches_oracle(gpu_lib, bits, dtype):
    wl = WORKLOADS["llama8b"]
    X = make_kv(wl, B=1, T=3000, which=0)[0, 1].to(dtype)  # one kv head: its outlier channels
    t, po, pr, perm = _setup(bits, X.float().numpy())
    n = X.shape[0]
    Ko, Kr = _lib.Records(n + 5, NO, NO, bits), _lib.Records(n + 5, D - NO, D - NO, bits - 1)
    _lib.tq_quantize_split(po, pr, perm, X.cuda(), Ko, Kr, out_offset=5)
    torch.cuda.synchronize()
    oO, oR = mixed.quantize_split(X.float().numpy(), t)
    for got_rec, oq, dim, w, bounds in ((Ko, oO, NO, bits, t.b_O), (Kr, oR, D - NO, bits - 1, t.b_R)):
        got = gpu_records_to_numpy(got_rec, slice(5, 5 + n), dim, dim, w)
        ok = check_indices(got["idx"], oq, bounds)
        check_signs(got["sgn"], oq, ok, dim)
        check_norms(got, oq, ok)


def _split_case(bits, B, Hq, Hkv, T, ctx, q_dtype, seed, own_records):
    """Keys and values with their own outlier channels (perm_k, perm_v)."""
    wl = WORKLOADS["llama8b"]
    K = make_kv(wl, B=B, T=T, which=0)[:, :Hkv].float()
    V = make_kv(wl, B=B, T=T, which=1)[:, :Hkv].float()
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g).to(q_dtype)
    t, po, pr, perm = _setup(bits, K[0, 0].numpy())
    t_v, _, _, perm_v = _setup(bits, V[0, 0].numpy())
    assert not np.array_equal(t.perm, t_v.perm)
    rows = B * Hkv * T
    Kf, Vf = K.reshape(rows, D).numpy(), V.reshape(rows, D).numpy()
    shape = lambda qq, dim: {"idx": qq.idx.reshape(B, Hkv, T, dim), "sgn": qq.sgn.reshape(B, Hkv, T, dim),
                             "norm": qq.norm.reshape(B, Hkv, T), "rnorm": qq.rnorm.reshape(B, Hkv, T)}
    if own_records:
        recs = []
        for X, pm in ((Kf, perm), (Vf, perm_v)):
            ro, rr = _lib.Records(rows, NO, NO, bits), _lib.Records(rows, D - NO, D - NO, bits - 1)
            _lib.tq_quantize_split(po, pr, pm, torch.from_numpy(X).cuda(), ro, rr)
            recs += [ro, rr]
        torch.cuda.synchronize()
        unp = [gpu_records_to_numpy(recs[i], slice(0, rows), dim, dim, w)
               for i, (dim, w) in enumerate(((NO, bits), (D - NO, bits - 1), (NO, bits), (D - NO, bits - 1)))]
        o_recs = []
        for u, dim in zip(unp, (NO, D - NO, NO, D - NO)):
            o_recs.append({"idx": u["idx"].reshape(B, Hkv, T, dim), "sgn": u["sgn"].reshape(B, Hkv, T, dim),
                           "norm": u["norm"].reshape(B, Hkv, T), "rnorm": u["rnorm"].reshape(B, Hkv, T)})
        Ko_g, Kr_g, Vo_g, Vr_g = recs
    else:
        kO, kR = mixed.quantize_split(Kf, t)
        vO, vR = mixed.quantize_split(Vf, t_v)
        o_recs = [shape(kO, NO), shape(kR, D - NO), shape(vO, NO), shape(vR, D - NO)]
        Ko_g, Kr_g = oracle_records_to_gpu(kO, NO, NO, bits), oracle_records_to_gpu(kR, D - NO, D - NO, bits - 1)
        Vo_g, Vr_g = oracle_records_to_gpu(vO, NO, NO, bits), oracle_records_to_gpu(vR, D - NO, D - NO, bits - 1)
    want, _ = mixed.decode_attention_split(q.float().numpy(), *o_recs, ctx, t, t_v=t_v)
    ws = torch.empty(_lib.tq_decode_split_workspace_size(po, pr, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    _lib.tq_decode_attention_split(po, pr, perm, perm_v, q.cuda(), Ko_g, Kr_g, Vo_g, Vr_g, ctx_t, T, Hkv, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), want


@pytest.mark.parametrize("bits", [2, 3])
def test_decode_split_on_oracle_records(gpu_lib, bits):
    out, want = _split_case(bits, 2, 8, 2, 700, [700, 333], torch.float32, 11 + bits, own_records=False)
    assert rel_l2(out, want) <= 1e-3


@pytest.mark.parametrize("bits", [2, 3])
def test_decode_split_on_gpu_records_bf16_query(gpu_lib, bits):
    out, want = _split_case(bits, 2, 8, 2, 1024, [1024, 1], torch.bfloat16, 21 + bits, own_records=True)
    assert rel_l2(out, want) <= 1e-3


def test_decode_split_empty_row_and_gqa8(gpu_lib):
    out, want = _split_case(2, 2, 8, 1, 300, [300, 0], torch.float32, 31, own_records=False)
    assert rel_l2(out[:1], want[:1]) <= 1e-3
    assert np.all(out[1] == 0.0)
