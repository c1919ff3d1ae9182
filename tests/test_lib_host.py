"""libturboquant on the host (no GPU): exports, setup tables vs the oracle, argument checks."""

import ctypes
import os
import re

import numpy as np
import pytest

from online_kv_cache_04_b300 import _lib
from oracle import codebook as ocb
from oracle import prng as oprng
from oracle import rotation as orot

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "turboquant.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:tq_status|size_t|int|const char\*)\s+(tq_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = _declared()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib._SIGNATURES)


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_rotation_matches_oracle(d):
    seed = 0x71550001
    got = _lib.tq_make_rotation(d, seed)
    want = orot.make_rotation(d, seed)
    tol = 1e-12 if d <= 128 else 2e-11  # Householder vs LAPACK: rounding grows with d·cond(G)
    assert np.abs(got - want).max() < tol


@pytest.mark.parametrize("d", [8, 32, 128, 1024])
@pytest.mark.parametrize("w", [1, 2, 3, 4])
def test_codebook_matches_oracle(d, w):
    c, b, mse = _lib.tq_make_codebook(d, w)
    oc, ob, omse, _ = ocb.lloyd_max(d, w)
    # relative to the outermost centroid: the oracle's incomplete-beta masses
    # carry ~1e-15 noise at d = 1024, which the fixed point amplifies to ~1e-13
    scale = np.abs(oc).max()
    assert np.abs(c - oc).max() < 1e-12 * scale
    assert np.abs(b - ob).max() < 1e-12 * scale
    assert abs(mse - omse) < 1e-12 / d


def test_qjl_matrix_matches_oracle_generator():
    m, d, seed = 64, 128, 0x71550002
    pi = orot.make_rotation(d, 0x71550001)
    S, s_rot = _lib.tq_make_qjl(m, d, seed, pi)
    So = oprng.gaussian_matrix(seed, m, d)
    assert np.abs(S - So).max() < 1e-13
    assert np.abs(s_rot - So @ pi.T).max() < 1e-12


def test_status_strings():
    lib = _lib.load()
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.tq_status_str(code)


def _fake_plan(d=128, m=128, w=2):
    """A plan whose device pointers are never dereferenced: only host checks run."""
    p = _lib.tq_plan()
    p.d, p.m, p.w = d, m, w
    for f in ("pi", "pi_t", "s_rot", "s_rot_t", "centroids", "bounds", "walsh", "pi_bf16", "s_bf16"):
        setattr(p, f, 4096)
    return p


def _fake_records(cap):
    return _lib.tq_records(4096, 8192, 12288, 16384, cap)


def test_argument_errors_return_codes_without_launching():
    lib = _lib.load()
    p = _fake_plan()
    r = _fake_records(100)
    ref = ctypes.byref
    # n < 0, beyond capacity, misaligned input, bad ld, bad dtype
    assert lib.tq_quantize(ref(p), 4096, 1, -1, 128, ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize(ref(p), 4096, 1, 90, 128, ref(r), 20, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize(ref(p), 4100, 1, 10, 128, ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize(ref(p), 4096, 1, 10, 100, ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize(ref(p), 4096, 7, 10, 128, ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize(ref(p), 4096, 1, 0, 128, ref(r), 0, None) == _lib.TQ_OK  # n = 0: no-op
    # the pair entry point checks both inputs and both outputs before any launch
    r2 = _fake_records(50)
    assert lib.tq_quantize_pair(ref(p), 4096, 8192, 1, 60, 128, ref(r), ref(r2), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize_pair(ref(p), 4096, 8200, 1, 10, 128, ref(r), ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize_pair(ref(p), 4096, None, 1, 10, 128, ref(r), ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize_pair(ref(p), 4096, 8192, 1, -1, 128, ref(r), ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize_pair(ref(p), 4096, 8192, 1, 10, 100, ref(r), ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize_pair(ref(p), 4096, 8192, 7, 10, 128, ref(r), ref(r), 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_quantize_pair(ref(p), 4096, 8192, 1, 0, 128, ref(r), ref(r2), 0, None) == _lib.TQ_OK
    # stage 1 alone: plans with m = 0 exist, and their records may omit signs and residual norms
    assert lib.tq_plan_bytes(128, 0, 2) > 0
    assert lib.tq_plan_bytes(128, 0, 2) < lib.tq_plan_bytes(128, 128, 2)
    nosig = _lib.tq_records(4096, None, 12288, None, 100)
    assert lib.tq_quantize(ref(p), 4096, 1, 10, 128, ref(nosig), 0, None) == _lib.TQ_ERR_ARG  # m = 128 needs them
    p0 = _fake_plan(128, 0, 2)
    assert lib.tq_quantize(ref(p0), 4096, 1, 0, 128, ref(nosig), 0, None) == _lib.TQ_OK
    assert lib.tq_quantize(ref(p0), 4096, 1, -1, 128, ref(nosig), 0, None) == _lib.TQ_ERR_ARG
    noidx = _lib.tq_records(None, None, 12288, None, 100)
    assert lib.tq_quantize(ref(p0), 4096, 1, 0, 128, ref(noidx), 0, None) == _lib.TQ_ERR_ARG
    # invalid plan shapes
    for d, m, w in ((100, 128, 2), (128, 128, 4), (2048, 128, 2), (128, 16, 2)):
        bad = _fake_plan(d, m, w)
        assert lib.tq_quantize(ref(bad), 4096, 1, 1, 128, ref(r), 0, None) == _lib.TQ_ERR_ARG
        assert lib.tq_plan_bytes(d, m, w) == 0
    # decode: Hq % Hkv, capacity, workspace
    n = ctypes.c_size_t(0)
    assert lib.tq_decode_workspace_size(ref(p), 1, 6, 4, 64, ref(n)) == _lib.TQ_ERR_ARG
    assert lib.tq_decode_workspace_size(ref(p), 1, 8, 2, 64, ref(n)) == _lib.TQ_OK and n.value > 0
    kv = _fake_records(2 * 64)
    args = (ref(p), 4096, 1, 1, 8, 2, ref(kv), ref(kv), 4096, 64, 0.0, 4096, 4096)
    assert lib.tq_decode_attention(*args, n.value - 4, None) == _lib.TQ_ERR_WORKSPACE
    small = _fake_records(2 * 64 - 1)
    assert lib.tq_decode_attention(ref(p), 4096, 1, 1, 8, 2, ref(small), ref(kv), 4096, 64, 0.0, 4096, 4096,
                                   n.value, None) == _lib.TQ_ERR_ARG
    assert lib.tq_decode_attention(ref(p), 4096, 1, 1, 6, 4, ref(kv), ref(kv), 4096, 64, 0.0, 4096, 4096,
                                   n.value, None) == _lib.TQ_ERR_ARG
    # decode limits: more than 8 query heads per kv head is unsupported
    big = _fake_records(64)
    assert lib.tq_decode_workspace_size(ref(p), 1, 16, 1, 64, ref(n)) == _lib.TQ_OK
    assert lib.tq_decode_attention(ref(p), 4096, 1, 1, 16, 1, ref(big), ref(big), 4096, 64, 0.0, 4096, 4096,
                                   n.value, None) == _lib.TQ_ERR_UNSUPPORTED
    # append: capacity, block-layout stride, dtype, shapes
    kv = _fake_records(2 * 64)
    kv2 = _lib.tq_records(20480, 24576, 28672, 32768, 2 * 64)
    assert lib.tq_append_kv(ref(p), 4096, 4096, 1, 1, 2, ref(kv), ref(kv), 4096, 64, None) == _lib.TQ_ERR_ARG
    assert lib.tq_append_kv(ref(p), 4096, 4096, 1, 1, 2, ref(kv), ref(kv2), 4096, 65, None) == _lib.TQ_ERR_ARG
    blk2 = _lib.tq_records(20480, 24576, 28672, 32768, 2 * 64, _lib.TQ_LAYOUT_BLOCK32)
    assert lib.tq_append_kv(ref(p), 4096, 4096, 1, 2, 1, ref(kv), ref(blk2), 4096, 48, None) == _lib.TQ_ERR_ARG
    assert lib.tq_append_kv(ref(p), 4096, 4096, 7, 1, 2, ref(kv), ref(kv2), 4096, 64, None) == _lib.TQ_ERR_ARG
    assert lib.tq_append_kv(ref(p), 4096, 4100, 1, 1, 2, ref(kv), ref(kv2), 4096, 64, None) == _lib.TQ_ERR_ARG
    assert lib.tq_append_kv(ref(p), 4096, 4096, 1, 0, 2, ref(kv), ref(kv2), 4096, 64, None) == _lib.TQ_ERR_ARG
    assert lib.tq_append_kv(ref(p), 4096, 4096, 1, 1, 2, ref(kv), ref(kv2), None, 64, None) == _lib.TQ_ERR_ARG
    assert lib.tq_append_kv(ref(p), 4096, 4096, 1, 1, 2, ref(kv), ref(kv2), 4096, 0, None) == _lib.TQ_ERR_ARG
    # decode with the fused append: the append's own checks, then the decode's, before any launch
    assert lib.tq_decode_workspace_size(ref(p), 1, 8, 2, 64, ref(n)) == _lib.TQ_OK
    app = lambda kn, vn, kvd, K, V, stride, pages, ws_bytes: lib.tq_decode_attention_append(
        ref(p), 4096, 1, kn, vn, kvd, 1, 8, 2, ref(K), ref(V), 4096, stride, pages, 0.0, 4096, 4096, ws_bytes, None)
    assert app(4096, 4096, 1, kv, kv, 64, None, n.value) == _lib.TQ_ERR_ARG      # K and V share their arrays
    assert app(4100, 4096, 1, kv, kv2, 64, None, n.value) == _lib.TQ_ERR_ARG     # misaligned new key
    assert app(4096, None, 1, kv, kv2, 64, None, n.value) == _lib.TQ_ERR_ARG     # no new value
    assert app(4096, 4096, 7, kv, kv2, 64, None, n.value) == _lib.TQ_ERR_ARG     # dtype
    assert app(4096, 4096, 1, kv, kv2, 64, 4096, n.value) == _lib.TQ_ERR_ARG     # pages need 256-token stride
    assert app(4096, 4096, 1, kv, kv2, 64, None, n.value - 4) == _lib.TQ_ERR_WORKSPACE
    # search: k range
    assert lib.tq_search_workspace_size(ref(p), 4, 100, 0, ref(n)) == _lib.TQ_ERR_ARG
    assert lib.tq_search_workspace_size(ref(p), 4, 100, 65, ref(n)) == _lib.TQ_ERR_ARG
    # setup
    assert lib.tq_make_rotation(1, 0, None) == _lib.TQ_ERR_ARG
    assert lib.tq_make_codebook(2, 1, None, None, None) == _lib.TQ_ERR_ARG


def test_layout_argument_checks():
    lib = _lib.load()
    p = _fake_plan()
    ref = ctypes.byref
    # block layout needs a capacity that is a multiple of 32; unknown layouts are rejected
    odd = _lib.tq_records(4096, 8192, 12288, 16384, 100, _lib.TQ_LAYOUT_BLOCK32)
    assert lib.tq_quantize(ref(p), 4096, 1, 10, 128, ref(odd), 0, None) == _lib.TQ_ERR_ARG
    bad = _lib.tq_records(4096, 8192, 12288, 16384, 128, 7)
    assert lib.tq_quantize(ref(p), 4096, 1, 10, 128, ref(bad), 0, None) == _lib.TQ_ERR_ARG
    rows = _lib.tq_records(4096, 8192, 12288, 16384, 2 * 64, _lib.TQ_LAYOUT_ROWS)
    blk = _lib.tq_records(4096, 8192, 12288, 16384, 2 * 64, _lib.TQ_LAYOUT_BLOCK32)
    n = ctypes.c_size_t(0)
    assert lib.tq_decode_workspace_size(ref(p), 1, 8, 2, 64, ref(n)) == _lib.TQ_OK
    # keys are read by vector: the block layout is refused for K
    assert lib.tq_decode_attention(ref(p), 4096, 1, 1, 8, 2, ref(blk), ref(blk), 4096, 64, 0.0, 4096, 4096,
                                   n.value, None) == _lib.TQ_ERR_UNSUPPORTED
    # block-layout values need ctx_stride % 32 == 0
    blk2 = _lib.tq_records(4096, 8192, 12288, 16384, 2 * 96, _lib.TQ_LAYOUT_BLOCK32)
    assert lib.tq_decode_workspace_size(ref(p), 1, 8, 2, 90, ref(n)) == _lib.TQ_OK
    rows2 = _lib.tq_records(4096, 8192, 12288, 16384, 2 * 96, _lib.TQ_LAYOUT_ROWS)
    assert lib.tq_decode_attention(ref(p), 4096, 1, 1, 8, 2, ref(rows2), ref(blk2), 4096, 90, 0.0, 4096, 4096,
                                   n.value, None) == _lib.TQ_ERR_ARG
    # search reads vectors: block layout unsupported
    assert lib.tq_search_workspace_size(ref(p), 4, 100, 10, ref(n)) == _lib.TQ_OK
    assert lib.tq_search_topk(ref(p), 4096, 1, 4, ref(blk), 100, 10, 4096, 4096, 4096, n.value,
                              None) == _lib.TQ_ERR_UNSUPPORTED


def test_binding_refuses_host_tensors_before_any_call():
    """A host pointer reaching a kernel would fault the GPU: the binding raises first."""
    import torch

    x = torch.zeros(4, 128)
    ctx = torch.zeros(1, dtype=torch.int32)
    rec = _lib.Records(64, 128, 128, 2, device="cpu")
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_quantize(None, x, rec)
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_quantize_pair(None, x, x, rec, rec)
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_append_kv(None, x[None], x[None], rec, rec, torch.zeros(1, dtype=torch.int32), 64)
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_decode_attention(None, x[None], rec, rec, ctx, 64, 1, x[None], torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_decode_attention_noalloc(None, x[None], rec, rec, ctx, 64, 1, x[None])
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_decode_scores(None, x[None], rec, ctx, 64, 1, x, torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        _lib.tq_search_topk(None, x, rec, 64, 10, torch.zeros(4, 10, dtype=torch.int32), torch.zeros(4, 10),
                            torch.zeros(16, dtype=torch.uint8))


@pytest.mark.parametrize("d", [4, 16, 128, 256])
def test_polar_codebooks_match_oracle(d):
    """The library's angle codebooks (uniform level 1, Lloyd-Max of sin^(k-1)(2ψ) later) against the oracle's."""
    from oracle import polar

    books, _, _ = _lib.tq_make_polar_codebooks(d)
    want = polar.make_codebooks(d)
    assert len(books) == len(want.books) == polar.levels(d)
    for (c, b), (wc, wb) in zip(books, want.books):
        assert np.allclose(c, wc, rtol=0, atol=1e-11)
        assert np.allclose(b, wb, rtol=0, atol=1e-11)
    assert _lib.load().tq_polar_index_words(d, 4, 2) == polar.index_words(d)
    assert _lib.load().tq_polar_index_words(96, 4, 2) == 0  # not a power of two
