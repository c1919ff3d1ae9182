"""The allocation-free decode entry point against the workspace one.

tq_decode_attention_noalloc serves callers that cannot allocate device
memory (graph captures that forbid allocation, embedded runtimes with memory
fixed at start-up, server plugins whose host owns the allocator): it takes
its scratch from an array compiled into the library instead of a caller
workspace.  Its results must equal tq_decode_attention's on the same records.
This file is collected last so that a failure here does not hide the others.
"""

import ctypes

import numpy as np
import pytest
import torch

from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_kv, make_queries

pytestmark = pytest.mark.gpu

TOL = 1e-3  # relative L2, the attention tolerance of the parity tests
SCRATCH_BYTES = 8 << 20


def _rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _cache(p, wl, B, Hkv, T, which, w):
    d = m = 128
    X = make_kv(wl, B=B, T=T, which=which)[:, :Hkv].contiguous().reshape(-1, d).cuda()
    rec = _lib.Records(B * Hkv * T, d, m, w)
    _lib.tq_quantize(p, X, rec)
    return rec


def test_noalloc_matches_workspace_entry_point_twice(gpu_lib):
    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED

    wl = WORKLOADS["llama8b"]
    d = m = 128
    w = 2
    p = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    B, Hq, Hkv, T = 2, 16, 4, 1500
    K = _cache(p, wl, B, Hkv, T, 0, w)
    V = _cache(p, wl, B, Hkv, T, 1, w)
    q = make_queries(wl, B=B)[:, :Hq].contiguous().cuda()
    ctx = torch.tensor([1500, 777], dtype=torch.int32, device="cuda")
    assert _lib.tq_decode_workspace_size(p, B, Hq, Hkv, T) <= SCRATCH_BYTES
    ws = torch.empty(_lib.tq_decode_workspace_size(p, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    want = torch.empty(B, Hq, d, device="cuda")
    _lib.tq_decode_attention(p, q, K, V, ctx, T, Hkv, want, ws)
    for call in range(2):  # the shared array keeps the previous call's contents
        got = torch.full((B, Hq, d), float("nan"), device="cuda")
        if call == 1:
            q = q * 0.5  # a different problem on the second call
            _lib.tq_decode_attention(p, q, K, V, ctx, T, Hkv, want, ws)
        _lib.tq_decode_attention_noalloc(p, q, K, V, ctx, T, Hkv, got)
        torch.cuda.synchronize()
        assert _rel_l2(got.cpu().numpy(), want.cpu().numpy()) <= TOL, call


def test_noalloc_rejects_shapes_beyond_its_scratch(gpu_lib):
    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED

    p = _lib.Plan(128, 128, 2, ROTATION_SEED, QJL_SEED)
    lib = _lib.load()
    B, Hq, Hkv, T = 4096, 64, 8, 1 << 20
    need = _lib.tq_decode_workspace_size(p, B, Hq, Hkv, T)
    assert need > SCRATCH_BYTES
    recs = _lib.tq_records(4096, 8192, 12288, 16384, B * Hkv * T)
    rc = lib.tq_decode_attention_noalloc(p.ref, 4096, _lib.TQ_BF16, B, Hq, Hkv, ctypes.byref(recs),
                                         ctypes.byref(recs), 4096, T, 0.0, 4096, None)
    assert rc == _lib.TQ_ERR_WORKSPACE
