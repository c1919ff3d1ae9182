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


# ---- 32-row block layout (value caches) -----------------------------------

def _run_block(X, d, m, w, offset, capacity, prefill=None):
    p = plan(d, m, w)
    rec = _lib.Records(capacity, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    rec.idx.fill_(-1 if prefill is None else prefill)
    rec.sgn.fill_(-1 if prefill is None else prefill)
    _lib.tq_quantize(p, X, rec, out_offset=offset)
    torch.cuda.synchronize()
    return rec


def _compare_block(X_host, rec, offset, d, m, w):
    from oracle import pack as opack

    n = X_host.shape[0]
    rows = np.arange(offset, offset + n)
    oq = oracle_quantize(X_host, d, m, w)
    got = gpu_records_to_numpy(rec, rows, d, m, w)
    _, _, _, bounds = oracle_tables(d, m, w)
    ok = check_indices(got["idx"], oq, bounds)
    check_signs(got["sgn"], oq, ok, d)
    check_norms(got, oq, ok)
    # whole blocks whose 32 rows all match: block words bit-identical to the oracle's packer
    iw = rec.idx.reshape(-1, w * d).cpu().numpy().view(np.uint32)
    sw = rec.sgn.reshape(-1, m).cpu().numpy().view(np.uint32)
    sg_ok = ok & np.all(got["sgn"] == oq.sgn, axis=1)
    checked = 0
    for b in range((offset + 31) // 32, (offset + n) // 32):
        sel = slice(32 * b - offset, 32 * b - offset + 32)
        if ok[sel].all():
            assert np.array_equal(iw[b], opack.pack_indices_block32(oq.idx[sel], w)[0])
            checked += 1
        if sg_ok[sel].all():
            assert np.array_equal(sw[b], opack.pack_signs_block32(oq.sgn[sel])[0])
    return oq, got, checked


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("n,off", [(4096, 0), (300, 64), (129, 0), (77, 5), (40, 60), (1, 31)])
def test_block_layout_bf16_tensor_core(gpu_lib, n, off, w):
    """bf16 d = m = 128: aligned rows on the tcgen05 kernel, a partial first block on the SIMT kernel."""
    wl = WORKLOADS["llama8b"]
    X = make_kv(wl, B=1, T=n, which=1)[0, (n + w) % 8]
    cap = ((off + n + 31) // 32 + 1) * 32
    rec = _run_block(X.cuda(), 128, 128, w, off, cap)
    _, _, checked = _compare_block(X.float().numpy(), rec, off, 128, 128, w)
    if n >= 64:
        assert checked > 0
    assert _lib.tq_fault_flags() == 0


def test_block_layout_merges_into_partly_written_blocks(gpu_lib):
    """Appending rows one call at a time keeps the other rows' bits of a block."""
    wl = WORKLOADS["llama8b"]
    d = m = 128
    w = 2
    X = make_kv(wl, B=1, T=100, which=0)[0, 2]
    p = plan(d, m, w)
    rec = _lib.Records(128, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    rec.idx.fill_(0x5A5A5A5A)
    rec.sgn.fill_(0x5A5A5A5A)
    Xd = X.cuda()
    for a, b in ((0, 3), (3, 4), (4, 37), (37, 70), (70, 100)):
        _lib.tq_quantize(p, Xd[a:b], rec, out_offset=a)
    torch.cuda.synchronize()
    _compare_block(X.float().numpy(), rec, 0, d, m, w)


@pytest.mark.parametrize("w", [1, 3])
def test_block_layout_fp32_simt(gpu_lib, w):
    wl = WORKLOADS["tiny"]
    K = make_kv(wl, which=1)[0, 0][:1000]
    rec = _run_block(K.cuda(), 128, 128, w, 24, 1024 + 32)
    _compare_block(K.numpy(), rec, 24, 128, 128, w)


@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("n,off,dtype", [(1000, 0, torch.bfloat16), (2048 + 77, 64, torch.bfloat16),
                                         (300, 20, torch.bfloat16), (500, 0, torch.float32)])
def test_quantize_pair_equals_two_calls(gpu_lib, w, n, off, dtype):
    """tq_quantize_pair (keys by row, values in 32-row blocks) gives bit-for-bit the records of
    two tq_quantize calls: one tensor-core launch for bf16 with a block-aligned offset, the two
    single calls otherwise (unaligned block offset, fp32 input).  The pair is checked against
    the oracle too."""
    d = m = 128
    wl = WORKLOADS["llama8b"]
    K = make_kv(wl, B=1, T=n, which=0, device="cuda").reshape(-1, d)[:n].to(dtype).contiguous()
    V = make_kv(wl, B=1, T=n, which=1, device="cuda").reshape(-1, d)[:n].to(dtype).contiguous()
    p = plan(d, m, w)
    cap = (n + off + 64 + 31) // 32 * 32  # block layout capacities are whole blocks
    outs = []
    for pair in (True, False):
        rk = _lib.Records(cap, d, m, w)
        rv = _lib.Records(cap, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
        for r in (rk, rv):
            r.idx.fill_(-1), r.sgn.fill_(-1), r.norm.fill_(-7.0), r.rnorm.fill_(-7.0)
        if pair:
            _lib.tq_quantize_pair(p, K, V, rk, rv, out_offset=off)
        else:
            _lib.tq_quantize(p, K, rk, out_offset=off)
            _lib.tq_quantize(p, V, rv, out_offset=off)
        torch.cuda.synchronize()
        assert _lib.tq_fault_flags() == 0
        outs.append([t.cpu().numpy() for r in (rk, rv) for t in (r.idx, r.sgn, r.norm, r.rnorm)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    rows = slice(off, off + n)
    rk = _lib.Records(cap, d, m, w)
    rv = _lib.Records(cap, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    _lib.tq_quantize_pair(p, K, V, rk, rv, out_offset=off)
    torch.cuda.synchronize()
    _compare(K.float().cpu().numpy(), rk, rows, d, m, w)
    _compare(V.float().cpu().numpy(), rv, rows, d, m, w)


@pytest.mark.parametrize("w", [1, 2, 3])
def test_wide_vectors_bf16_ragged_offset(gpu_lib, w):
    """d = m = 512 bf16 input, 1000 vectors (not a multiple of the 16-vector tile) written at row 37
    of a 1100-row cache: indices, signs and norms against the oracle, other rows untouched."""
    d = 512
    g = torch.Generator().manual_seed(500 + w)
    X = (torch.randn(1000, d, generator=g) * (1 + 9 * (torch.rand(d, generator=g) < 0.03))).to(torch.bfloat16)
    rec = _run(X.cuda(), d, d, w, offset=37, capacity=1100)
    _compare(X.float().numpy(), rec, slice(37, 1037), d, d, w)
    assert bool((rec.idx[:37] == -1).all()) and bool((rec.idx[1037:] == -1).all())
    assert bool((rec.sgn[:37] == -1).all()) and bool((rec.sgn[1037:] == -1).all())


@pytest.mark.parametrize("w,m", [(2, 128), (3, 128), (2, 0)])
def test_pair_repeated_launches_full_layer(gpu_lib, w, m):
    """The paired tensor-core launch over a whole Llama-3.1-8B-shaped layer (2 x 262,144
    vectors: 28 tiles for most CTAs, so the warp roles run several tiles apart) repeated 40
    times: no bounded wait runs out and every launch writes the same records, bit for bit.
    Rows sampled across the layer match the oracle."""
    d = 128
    wl = WORKLOADS["llama8b"]
    n = wl.B * wl.Hkv * wl.ctx
    K = make_kv(wl, which=0, device="cuda").reshape(n, d)
    V = make_kv(wl, which=1, device="cuda").reshape(n, d)
    p = plan(d, m, w)
    rk = _lib.Records(n, d, m, w)
    rv = _lib.Records(n, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    _lib.tq_fault_flags(reset=True)
    _lib.tq_quantize_pair(p, K, V, rk, rv)
    torch.cuda.synchronize()
    fields = lambda: [t.clone() for r in (rk, rv) for t in (r.idx, r.sgn, r.norm, r.rnorm) if t is not None]
    first = fields()
    for _ in range(40):
        _lib.tq_quantize_pair(p, K, V, rk, rv)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags() == 0
    for a, b in zip(first, fields()):
        assert torch.equal(a, b)
    for r0 in (0, n // 2 + 32, n - 64):  # block-aligned ranges at the start, middle and end
        rows = slice(r0, r0 + 64)
        _compare(K[rows].float().cpu().numpy(), rk, rows, d, m, w)
        _compare(V[rows].float().cpu().numpy(), rv, rows, d, m, w)
