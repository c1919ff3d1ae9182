"""GPU parity of the wide-vector tcgen05 quantizer (d a multiple of 256 up to
1024, m = d or 0, records by row) against the float64 oracle.

Its sign stage forms S r / n as S x / n - (S Πᵀ) c[idx] rather than from the
residual ("谷歌TurboQuant如何绕过内存墙？" §2 stage 2: σ = sign(S r)); the sign,
index and norm rules of tests/parity.py are the same as for every other path.
Cases span one tile and many (several 128-vector tiles per CTA, so the
persistent loop's barrier phases turn over), ragged tails, output offsets,
zero vectors and both input types.
"""

import numpy as np
import pytest
import torch

from online_kv_cache_04_b300 import _lib
from online_kv_cache_04_b300.workloads import WORKLOADS, make_generic

from parity import (check_indices, check_norms, check_signs, gpu_records_to_numpy, oracle_quantize, oracle_tables,
                    plan)

pytestmark = pytest.mark.gpu


def _inputs(n, d, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(n, d, generator=g) * (1 + 9 * (torch.rand(d, generator=g) < 0.03))
    return X.to(dtype)


def _quantize(X, d, m, w, offset=0, capacity=None):
    p = plan(d, m, w)
    n = X.shape[0]
    rec = _lib.Records(capacity or n + offset, d, m, w)
    rec.idx.fill_(-1)
    if m > 0:
        rec.sgn.fill_(-1)
    _lib.tq_quantize(p, X.cuda(), rec, out_offset=offset)
    torch.cuda.synchronize()
    assert _lib.tq_fault_flags(reset=True) == 0
    return rec


def _check(X_host, rec, rows, d, m, w):
    from oracle import pack as opack

    oq = oracle_quantize(X_host, d, m, w)
    got = gpu_records_to_numpy(rec, rows, d, m, w)
    _, _, _, bounds = oracle_tables(d, m, w)
    ok = check_indices(got["idx"], oq, bounds)
    assert np.array_equal(got["idx_words"][ok], opack.pack_indices(oq.idx[ok], w))
    if m > 0:
        check_signs(got["sgn"], oq, ok, d)
        sg_ok = ok & np.all(got["sgn"] == oq.sgn, axis=1)
        assert np.array_equal(got["sgn_words"][sg_ok], opack.pack_signs(oq.sgn[sg_ok]))
    check_norms(got, oq, ok)
    return oq, got


@pytest.mark.parametrize("d", [256, 512, 768, 1024])
@pytest.mark.parametrize("w", [1, 2, 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_two_stage_matches_oracle(gpu_lib, d, w, dtype):
    """300 vectors (three tiles, the last ragged) written at row 5 of a 320-row array."""
    X = _inputs(300, d, 7000 + d + 10 * w + (dtype == torch.bfloat16), dtype)
    rec = _quantize(X, d, d, w, offset=5, capacity=320)
    _check(X.float().numpy(), rec, slice(5, 305), d, d, w)
    assert bool((rec.idx[:5] == -1).all()) and bool((rec.idx[305:] == -1).all())
    assert bool((rec.sgn[:5] == -1).all()) and bool((rec.sgn[305:] == -1).all())


@pytest.mark.parametrize("d,w", [(256, 3), (512, 2), (1024, 3)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_stage1_alone_matches_oracle(gpu_lib, d, w, dtype):
    """m = 0: indices and norms only ("谷歌TurboQuant如何绕过内存墙？" §2 stage 1)."""
    X = _inputs(129, d, 7100 + d + w, dtype)
    rec = _quantize(X, d, 0, w)
    _check(X.float().numpy(), rec, slice(0, 129), d, 0, w)


@pytest.mark.parametrize("n", [1, 127, 128, 129])
def test_one_tile_edges(gpu_lib, n):
    X = _inputs(n, 1024, 7200 + n)
    rec = _quantize(X, 1024, 1024, 3)
    _check(X.numpy(), rec, slice(0, n), 1024, 1024, 3)


def test_zero_and_large_vectors(gpu_lib):
    """A zero vector (indices of u = 0, all sign bits set, zero norms) and rows
    scaled by 1e-6 and 1e6 (only the direction matters) beside ordinary ones."""
    d = 512
    X = _inputs(200, d, 7300)
    X[3] = 0.0
    X[4] *= 1e-6
    X[5] *= 1e6
    X[130] = 0.0
    rec = _quantize(X, d, d, 3)
    _check(X.numpy(), rec, slice(0, 200), d, d, 3)
    for r in (3, 130):
        assert float(rec.norm[r]) == 0.0 and float(rec.rnorm[r]) == 0.0
        assert bool((rec.sgn[r] == -1).all())


def test_many_tiles_per_cta_sampled(gpu_lib):
    """2.5 tiles per SM at d = 256: the persistent loop turns every ring and
    accumulator slot over many times; the oracle checks every 16th row."""
    d = 256
    n = 148 * 128 * 2 + 128 * 60 + 77
    X = _inputs(n, d, 7400)
    rec = _quantize(X, d, d, 2)
    rows = np.arange(0, n, 16)
    rows[-1] = n - 1
    _check(X[rows].numpy(), rec, torch.as_tensor(rows, device="cuda"), d, d, 2)


def test_generic_full_size_sampled(gpu_lib):
    """The generic workload at full size: 1,048,576 unit-norm anisotropic fp32
    vectors, d = m = 1024, b = 4; the oracle checks 4096 rows spread over it."""
    wl = WORKLOADS["generic"]
    X = make_generic(wl, n=wl.ctx, device="cuda")
    rec = _quantize(X, 1024, 1024, 3)
    rows = torch.arange(0, wl.ctx, 256)
    rows[-1] = wl.ctx - 1
    _check(X[rows.cuda()].cpu().numpy(), rec, rows, 1024, 1024, 3)


@pytest.mark.parametrize("d", [384, 640, 896])
def test_warp_mma_quantizer_at_odd_multiples_of_128(gpu_lib, d):
    """Multiples of 128 that are not multiples of 256 take the warp-MMA kernel,
    whose warps then own d/8 coordinates rounded up to whole index words."""
    X = _inputs(257, d, 7500 + d)
    rec = _quantize(X, d, d, 3)
    _check(X.numpy(), rec, slice(0, 257), d, d, 3)
