"""The allocation-free decode entry point against the workspace one.

tq_decode_attention_noalloc serves callers that cannot allocate device
memory (graph captures that forbid allocation, embedded runtimes with memory
fixed at start-up, server plugins whose host owns the allocator): it takes
its scratch from an array compiled into the library instead of a caller
workspace.  Its results must equal tq_decode_attention's on the same records,
including when the array still holds what an earlier call of another shape
left there.  This file is collected last so that a failure here does not hide
the others.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_kv, make_queries

from parity import oracle_quantize, oracle_records_to_gpu, oracle_tables, plan, rel_l2

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20
BLK = _lib.TQ_LAYOUT_BLOCK32


def _cache(p, wl, B, Hkv, T, which, w, layout=_lib.TQ_LAYOUT_ROWS):
    d = m = 128
    X = make_kv(wl, B=B, T=T, which=which)[:, :Hkv].contiguous().reshape(-1, d).cuda()
    rec = _lib.Records(B * Hkv * T, d, m, w, layout=layout)
    _lib.tq_quantize(p, X, rec)
    return rec


def _with_workspace(p, q, K, V, ctx, T, Hkv):
    B, Hq, d = q.shape
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention(p, q, K, V, ctx, T, Hkv, out, ws)
    return out


def _without(p, q, K, V, ctx, T, Hkv):
    B, Hq, d = q.shape
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    _lib.tq_decode_attention_noalloc(p, q, K, V, ctx, T, Hkv, out)
    return out


def test_noalloc_general_path_equals_workspace_entry_point_twice(gpu_lib):
    """Values in the row layout and T not a multiple of 128: the general split/combine kernels.

    Same kernels, same inputs, no atomics in the arithmetic: the results must be
    bit-identical, on two calls in a row with different problems."""
    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED

    wl = WORKLOADS["llama8b"]
    w = 2
    p = _lib.Plan(128, 128, w, ROTATION_SEED, QJL_SEED)
    B, Hq, Hkv, T = 2, 16, 4, 1500
    K = _cache(p, wl, B, Hkv, T, 0, w)
    V = _cache(p, wl, B, Hkv, T, 1, w)
    q = make_queries(wl, B=B)[:, :Hq].contiguous().cuda()
    ctx = torch.tensor([1500, 777], dtype=torch.int32, device="cuda")
    assert _lib.tq_decode_workspace_size(p, B, Hq, Hkv, T) <= SCRATCH_BYTES
    for call in range(2):  # the shared array keeps the previous call's contents
        if call == 1:
            q = q * 0.5  # a different problem on the second call
        want = _with_workspace(p, q, K, V, ctx, T, Hkv)
        got = _without(p, q, K, V, ctx, T, Hkv)
        torch.cuda.synchronize()
        assert _lib.tq_fault_flags() == 0
        assert torch.equal(got, want), call


def test_noalloc_tensor_core_path_after_a_larger_call(gpu_lib):
    """Values in 32-row blocks and T a multiple of 128: the tensor-core decode.

    That path keeps per-unit query tables and per-unit arrival counters in the
    scratch.  A larger no-alloc call first fills the array with tables and
    counters of another unit count; the smaller call that follows must still
    match the workspace entry point and the float64 oracle.  Both entry points
    run the same kernels; the query-table kernel sums four warps' offset terms
    with float atomics, whose order may change the last bits of a score
    constant between two calls, so the two outputs are compared at 1e-6
    relative L2 rather than bit for bit."""
    d = m = 128
    w = 2
    p = plan(d, m, w)
    g = torch.Generator().manual_seed(77)
    # the larger shape: 4 x 8 units of 2048 tokens, every CTA busy
    Bb, Hqb, Hkvb, Tb = 4, 32, 8, 2048
    Kb = torch.randn(Bb * Hkvb * Tb, d, generator=g).cuda()
    Vb = torch.randn(Bb * Hkvb * Tb, d, generator=g).cuda()
    Kbr = _lib.Records(Bb * Hkvb * Tb, d, m, w)
    Vbr = _lib.Records(Bb * Hkvb * Tb, d, m, w, layout=BLK)
    _lib.tq_quantize(p, Kb, Kbr)
    _lib.tq_quantize(p, Vb, Vbr)
    qb = torch.randn(Bb, Hqb, d, generator=g).cuda()
    ctxb = torch.full((Bb,), Tb, dtype=torch.int32, device="cuda")
    assert _lib.tq_decode_workspace_size(p, Bb, Hqb, Hkvb, Tb) <= SCRATCH_BYTES
    big = _without(p, qb, Kbr, Vbr, ctxb, Tb, Hkvb)
    torch.cuda.synchronize()
    assert torch.isfinite(big).all()

    # the smaller shape on the oracle's own records, ragged second row
    B, Hq, Hkv, T = 2, 8, 2, 1536
    ctx = [1536, 700]
    K = torch.randn(B, Hkv, T, d, generator=g)
    V = torch.randn(B, Hkv, T, d, generator=g)
    q = torch.randn(B, Hq, d, generator=g)
    kq = oracle_quantize(K.numpy().reshape(-1, d), d, m, w)
    vq = oracle_quantize(V.numpy().reshape(-1, d), d, m, w)
    shape = lambda oq: {"idx": oq.idx.reshape(B, Hkv, T, d), "sgn": oq.sgn.reshape(B, Hkv, T, m),
                        "norm": oq.norm.reshape(B, Hkv, T), "rnorm": oq.rnorm.reshape(B, Hkv, T)}
    Pi, S, c, _ = oracle_tables(d, m, w)
    oracle_out, _ = odec.decode_attention(q.numpy(), shape(kq), shape(vq), ctx, Pi, S, c)
    Kr = oracle_records_to_gpu(kq, d, m, w)
    Vr = oracle_records_to_gpu(vq, d, m, w, layout=BLK)
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    qg = q.cuda()
    for call in range(2):
        got = _without(p, qg, Kr, Vr, ctx_t, T, Hkv)
        want = _with_workspace(p, qg, Kr, Vr, ctx_t, T, Hkv)
        torch.cuda.synchronize()
        assert _lib.tq_fault_flags() == 0
        got, want = got.cpu().numpy(), want.cpu().numpy()
        assert rel_l2(got, want) <= 1e-6, call
        assert rel_l2(got, oracle_out) <= 1e-3, call


def test_noalloc_rejects_shapes_beyond_its_scratch(gpu_lib):
    """A shape whose workspace exceeds the array is refused on the host, before any launch."""
    w = 2
    p = plan(128, 128, w)
    B, Hq, Hkv, T = 4096, 64, 8, 1 << 20
    assert _lib.tq_decode_workspace_size(p, B, Hq, Hkv, T) > SCRATCH_BYTES
    # small real buffers: the size check must refuse the call before anything reads them
    K = _lib.Records(32, 128, 128, w)
    V = _lib.Records(32, 128, 128, w, layout=BLK)
    K.c.capacity = V.c.capacity = B * Hkv * T  # the shape the call claims
    q = torch.zeros(1, Hq, 128, device="cuda")
    out = torch.zeros(1, Hq, 128, device="cuda")
    ctx = torch.zeros(B, dtype=torch.int32, device="cuda")
    rc = _lib.load().tq_decode_attention_noalloc(p.ref, q.data_ptr(), _lib.TQ_F32, B, Hq, Hkv, K.ref, V.ref,
                                                 ctx.data_ptr(), T, 0.0, out.data_ptr(), None)
    assert rc == _lib.TQ_ERR_WORKSPACE
    assert torch.equal(out, torch.zeros_like(out))
