"""GPU parity of tq_quantize against the float64 oracle (through the C ABI)."""

import numpy as np
import pytest
import torch

from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_generic, make_kv

from parity import (check_indices, check_norms, check_signs, gpu_records_to_numpy, oracle_quantize, oracle_tables,
                    plan)

pytestmark = pytest.mark.gpu


def _run(X, d, m, w, offset=0, capacity=None):
    p = plan(d, m, w)
    n = X.shape[0]
    rec = _lib.Records(capacity or n + offset, d, m, w)
    rec.idx.fill_(-1)
    rec.sgn.fill_(-1)
    _lib.tq_quantize(p, X, rec, out_offset=offset)
    torch.cuda.synchronize()
    return rec


def _compare(X_host, rec, rows, d, m, w):
    oq = oracle_quantize(X_host, d, m, w)
    got = gpu_records_to_numpy(rec, rows, d, m, w)
    _, _, _, bounds = oracle_tables(d, m, w)
    ok = check_indices(got["idx"], oq, bounds)
    check_signs(got["sgn"], oq, ok, d)
    check_norms(got, oq, ok)
    # packing: fully matching vectors are bit-identical to the oracle's packed words
    from oracle import pack as opack

    want_words = opack.pack_indices(oq.idx[ok], w)
    assert np.array_equal(got["idx_words"][ok], want_words)
    sg_ok = ok & np.all(got["sgn"] == oq.sgn, axis=1)
    assert np.array_equal(got["sgn_words"][sg_ok], opack.pack_signs(oq.sgn[sg_ok]))
    return oq, got


@pytest.mark.parametrize("w", [1, 2, 3])
def test_tiny_workload_fp32(gpu_lib, w):
    wl = WORKLOADS["tiny"]
    K = make_kv(wl, which=0)[0, 0]  # [4096, 128] fp32, outlier channels x10
    rec = _run(K.cuda(), 128, 128, w)
    _compare(K.numpy(), rec, slice(0, K.shape[0]), 128, 128, w)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 33, 1000])
def test_ragged_counts_and_append_offset(gpu_lib, n):
    g = torch.Generator().manual_seed(n)
    X = torch.randn(n, 128, generator=g)
    off = 7
    rec = _run(X.cuda(), 128, 128, 2, offset=off, capacity=n + off + 5)
    _compare(X.numpy(), rec, slice(off, off + n), 128, 128, 2)
    # rows outside [off, off + n) untouched
    assert torch.all(rec.idx[:off] == -1) and torch.all(rec.idx[off + n:] == -1)


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("n", [1, 127, 128, 129, 300, 2000])
def test_bf16_tensor_core_path_ragged_and_offset(gpu_lib, n, w):
    """bf16, d = m = 128 runs on the tcgen05 kernel: tails of every tile size, append offset."""
    wl = WORKLOADS["llama8b"]
    X = make_kv(wl, B=1, T=n, which=0)[0, n % 8]  # bf16 [n, 128]
    off = 5
    rec = _run(X.cuda(), 128, 128, w, offset=off, capacity=n + off + 3)
    _compare(X.float().numpy(), rec, slice(off, off + n), 128, 128, w)
    assert torch.all(rec.idx[:off] == -1) and torch.all(rec.idx[off + n:] == -1)
    assert torch.all(rec.sgn[:off] == -1) and torch.all(rec.sgn[off + n:] == -1)
    assert _lib.tq_fault_flags() == 0


def test_zero_vector_and_bf16_input(gpu_lib):
    wl = WORKLOADS["llama8b"]
    X = make_kv(wl, B=1, T=64, which=1)[0, 3]  # bf16 [64, 128]
    X[5] = 0
    rec = _run(X.cuda(), 128, 128, 3)
    oq, got = _compare(X.float().numpy(), rec, slice(0, 64), 128, 128, 3)
    assert got["norm"][5] == 0 and got["rnorm"][5] == 0 and got["sgn"][5].all()


def test_strided_rows(gpu_lib):
    X = torch.randn(300, 136)
    Xd = X.cuda()[:, :128]
    assert Xd.stride(0) == 136
    rec = _run(Xd, 128, 128, 2)  # leading dimension 136
    _compare(X[:, :128].numpy(), rec, slice(0, 300), 128, 128, 2)


@pytest.mark.parametrize("d,w", [(32, 1), (64, 3), (256, 2), (1024, 3)])
def test_other_dims(gpu_lib, d, w):
    g = torch.Generator().manual_seed(d)
    X = torch.randn(257, d, generator=g) * (1 + 9 * (torch.rand(d, generator=g) < 0.03))
    rec = _run(X.cuda(), d, d, w)
    _compare(X.numpy(), rec, slice(0, 257), d, d, w)


def test_prefill_full_size_sampled(gpu_lib):
    """8 kv heads x 65536 tokens x {K, V}, bf16, b = 3; oracle on 8192 sampled rows."""
    wl = WORKLOADS["prefill"]
    K = make_kv(wl, which=0, device="cuda")[0]  # [8, 65536, 128] bf16
    V = make_kv(wl, which=1, device="cuda")[0]
    X = torch.cat([K.reshape(-1, 128), V.reshape(-1, 128)])
    del K, V
    rec = _run(X, 128, 128, 2)
    rows = torch.randperm(X.shape[0], generator=torch.Generator().manual_seed(4))[:8192].sort().values
    _compare(X[rows.cuda()].float().cpu().numpy(), rec, rows, 128, 128, 2)


def test_generic_d1024_sampled(gpu_lib):
    """Unit-norm anisotropic fp32 vectors, d = m = 1024, b = 4 (65536-vector slice)."""
    wl = WORKLOADS["generic"]
    X = make_generic(wl, n=65536, device="cuda")
    rec = _run(X, 1024, 1024, 3)
    rows = torch.arange(0, 65536, 64)
    _compare(X[rows.cuda()].cpu().numpy(), rec, rows, 1024, 1024, 3)
