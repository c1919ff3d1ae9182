"""Pins for the oracle's quantizer, QJL estimator and packing (no GPU)."""

import math

import numpy as np
import pytest

from oracle import codebook, pack, prng, qjl, quantize, rotation


def _setup(d, w, m=None, rs=11, qs=22):
    m = d if m is None else m
    Pi = rotation.make_rotation(d, rs)
    S = qjl.make_qjl(m, d, qs)
    c, b, mse, _ = codebook.lloyd_max(d, w)
    return Pi, S, c, b, mse


@pytest.mark.parametrize("w", [1, 2, 3])
def test_bucketize_is_brute_force_nearest_codeword(w):
    d = 8
    Pi, S, c, b, _ = _setup(d, w)
    X = prng.normals(3, 4000 * d).reshape(4000, d)
    q = quantize.quantize(X, Pi, S, c, b)
    dist = np.abs(q.u[..., None] - c[None, None, :])
    nearest = np.argmin(dist, axis=-1)
    sorted_d = np.sort(dist, axis=-1)
    clear = (sorted_d[..., 1] - sorted_d[..., 0]) > 1e-12
    assert clear.mean() > 0.999
    assert np.array_equal(q.idx[clear], nearest[clear])


@pytest.mark.parametrize("w", [1, 2, 3])
def test_vectors_on_a_codeword_ray(w):
    """x = t·Πᵀc[idx]: u = c[idx]/‖c[idx]‖ keeps idx, x̃ = ‖x‖Πᵀc[idx], so
    ‖r‖ = t·‖c[idx]‖·|1 - ‖c[idx]‖| and r is parallel to x."""
    d = 32
    Pi, S, c, b, _ = _setup(d, w)
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 1 << w, size=(50, d))
    cn = np.linalg.norm(c[idx], axis=1)
    # keep rows where c[idx]/‖c[idx]‖ stays strictly inside every cell
    lo = np.concatenate([[-np.inf], b])[idx]
    hi = np.concatenate([b, [np.inf]])[idx]
    v = c[idx] / cn[:, None]
    keep = np.all((v > lo + 1e-9) & (v < hi - 1e-9), axis=1)
    idx, cn = idx[keep], cn[keep]
    assert len(idx) > 5
    t = 2.0 ** rng.integers(-3, 4, size=len(idx))
    X = t[:, None] * (c[idx] @ Pi)
    q = quantize.quantize(X, Pi, S, c, b)
    assert np.array_equal(q.idx, idx)
    assert np.allclose(q.norm, t * cn, rtol=1e-7, atol=0)
    assert np.allclose(q.rnorm64, t * cn * np.abs(1.0 - cn), rtol=1e-9, atol=1e-14)


def test_zero_vector_rule():
    d, w = 32, 2
    Pi, S, c, b, _ = _setup(d, w)
    q = quantize.quantize(np.zeros((1, d)), Pi, S, c, b)
    # u = 0 lies on the middle boundary 0: #{β < 0} = 1 (tie -> lower cell)
    assert np.all(q.idx == 1)
    assert q.norm[0] == 0 and q.rnorm[0] == 0 and q.sgn.all()


@pytest.mark.parametrize("w", [1, 2, 3])
def test_stage1_distortion_matches_codebook_and_printed_bounds(w):
    d, N = 128, 20000
    Pi, S, c, b, mse = _setup(d, w)
    X = prng.normals(77, N * d).reshape(N, d)
    X /= np.linalg.norm(X, axis=1, keepdims=True)
    _, _, _, xt = quantize.stage1(X, Pi, c, b)
    err = np.sum((X - xt) ** 2, axis=1)
    se = err.std() / math.sqrt(N)
    assert abs(err.mean() - d * mse) < 4 * se
    assert 4.0 ** -w <= err.mean() <= math.sqrt(3) * math.pi / 2 * 4.0 ** -w


def test_one_bit_mse_quantizer_shrinks_inner_products_toward_2_over_pi():
    """E⟨x, x̃⟩ / ‖x‖² = d·c² (exact), which tends to 2/π ≈ 0.637 as d grows."""
    gaps = []
    for d in (128, 1024):
        Pi, S, c, b, _ = _setup(d, 1)
        N = 4000
        X = prng.normals(d, N * d).reshape(N, d)
        X /= np.linalg.norm(X, axis=1, keepdims=True)
        _, _, _, xt = quantize.stage1(X, Pi, c, b)
        ratio = np.sum(X * xt, axis=1)
        exact = d * c[1] ** 2
        assert abs(ratio.mean() - exact) < 4 * ratio.std() / math.sqrt(N) + 1e-12
        gaps.append(abs(exact - 2 / math.pi))
    assert gaps[1] < gaps[0] and gaps[1] < 5e-4


def test_qjl_estimator_unbiased_with_closed_form_variance():
    d = m = 32
    rng = np.random.default_rng(5)
    q = rng.standard_normal(d)
    r = rng.standard_normal(d)
    est = []
    for s in range(10000):
        S = qjl.make_qjl(m, d, 500000 + s)
        est.append(qjl.estimate(S, q, np.linalg.norm(r), qjl.signs(S, r)))
    est = np.array(est)
    truth = q @ r
    se = est.std() / math.sqrt(len(est))
    assert abs(est.mean() - truth) < 3 * se
    var = ((math.pi / 2) * (q @ q) * (r @ r) - truth ** 2) / m
    assert abs(est.var() / var - 1.0) < 0.05


def test_two_stage_score_is_unbiased_over_S():
    """Stage 1 + QJL on the residual: E_S[⟨q, x̂⟩] = ⟨q, x⟩ -- for a random q, and
    for q along the residual r = x - x̃ (not a function of S), where the QJL
    term carries the whole correction and any error in its scale shows."""
    d = m = 32
    w = 1
    Pi = rotation.make_rotation(d, 3)
    c, b, _, _ = codebook.lloyd_max(d, w)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, d))
    _, _, _, xt = quantize.stage1(x, Pi, c, b)
    r = x[0] - xt[0]
    qs = np.stack([rng.standard_normal(d), r / np.linalg.norm(r)])
    vals = []
    for s in range(10000):
        S = qjl.make_qjl(m, d, 900000 + s)
        z = quantize.quantize(x, Pi, S, c, b)
        xh = quantize.reconstruct(z.idx, z.sgn, z.norm, z.rnorm, Pi, S, c)
        vals.append(qs @ xh[0])
    vals = np.array(vals)
    se = vals.std(axis=0) / math.sqrt(len(vals))
    # fp32 storage of the norms biases by at most ~1e-7 relative
    assert np.all(np.abs(vals.mean(axis=0) - qs @ x[0]) < 3 * se + 1e-6)


def test_reconstruct_inner_product_is_the_estimator():
    d, w = 64, 2
    Pi, S, c, b, _ = _setup(d, w)
    rng = np.random.default_rng(1)
    X = rng.standard_normal((5, d))
    qv = rng.standard_normal(d)
    z = quantize.quantize(X, Pi, S, c, b)
    xh = quantize.reconstruct(z.idx, z.sgn, z.norm, z.rnorm, Pi, S, c)
    for i in range(5):
        mse_part = float(z.norm[i]) * float(c[z.idx[i]] @ (Pi @ qv))
        sig = np.where(z.sgn[i], 1.0, -1.0)
        est = mse_part + qjl.estimate(S, qv, float(z.rnorm[i]), sig)
        assert abs(xh[i] @ qv - est) < 1e-12 * (1 + abs(est))


# ---- packing ---------------------------------------------------------------

def test_pack_hand_patterns():
    d = 64
    j = np.arange(d)
    # w = 2, idx = j mod 4: plane 0 = odd j, plane 1 = j mod 4 in {2, 3}
    words = pack.pack_indices((j % 4)[None, :], 2)[0]
    assert [int(x) for x in words] == [0xAAAAAAAA, 0xAAAAAAAA, 0xCCCCCCCC, 0xCCCCCCCC]
    # w = 3, idx = j mod 8
    words = pack.pack_indices((j % 8)[None, :], 3)[0]
    assert [int(x) for x in words] == [0xAAAAAAAA] * 2 + [0xCCCCCCCC] * 2 + [0xF0F0F0F0] * 2
    # all zero / all ones
    assert not pack.pack_indices(np.zeros((1, d), int), 3).any()
    assert np.all(pack.pack_indices(np.full((1, d), 7), 3) == 0xFFFFFFFF)
    # idx = 1 only at coordinate 33 -> plane 0, word 1, bit 1
    idx = np.zeros((1, d), int)
    idx[0, 33] = 1
    assert [int(x) for x in pack.pack_indices(idx, 2)[0]] == [0, 2, 0, 0]
    # signs: +1 at even j -> 0x55555555
    assert [int(x) for x in pack.pack_signs((j % 2 == 0)[None, :])[0]] == [0x55555555, 0x55555555]


@pytest.mark.parametrize("w", [1, 2, 3])
def test_pack_round_trip(w):
    rng = np.random.default_rng(w)
    idx = rng.integers(0, 1 << w, size=(7, 96))
    sg = rng.integers(0, 2, size=(7, 128)).astype(bool)
    assert np.array_equal(pack.unpack_indices(pack.pack_indices(idx, w), w, 96), idx)
    assert np.array_equal(pack.unpack_signs(pack.pack_signs(sg)), sg)


def test_pack_block32_hand_patterns():
    d, w = 64, 2
    idx = np.zeros((64, d), int)
    idx[1, 5] = 1           # block 0, row 1 -> bit 16 of plane-0 word 5
    idx[2, 5] = 2           # block 0, row 2 -> bit 1 of plane-1 word 5
    idx[32 + 31, 63] = 3    # block 1, row 31 -> bit 31 of both planes' word 63
    words = pack.pack_indices_block32(idx, w)
    assert words.shape == (2, w * d)
    expect = np.zeros((2, w * d), np.uint64)
    expect[0, 5] = 1 << 16
    expect[0, d + 5] = 1 << 1
    expect[1, 63] = 1 << 31
    expect[1, d + 63] = 1 << 31
    assert np.array_equal(words, expect.astype(np.uint32))
    # every even row set -> low half-word full; every odd row -> high half
    sg = np.zeros((32, 32), bool)
    sg[0::2, 0] = True
    sg[1::2, 1] = True
    sw = pack.pack_signs_block32(sg)[0]
    assert int(sw[0]) == 0x0000FFFF and int(sw[1]) == 0xFFFF0000 and not sw[2:].any()


@pytest.mark.parametrize("w", [1, 2, 3])
def test_pack_block32_round_trip_and_transpose_of_row_layout(w):
    rng = np.random.default_rng(10 + w)
    N, d, m = 96, 64, 96
    idx = rng.integers(0, 1 << w, size=(N, d))
    sg = rng.integers(0, 2, size=(N, m)).astype(bool)
    bw = pack.pack_indices_block32(idx, w)
    assert np.array_equal(pack.unpack_indices_block32(bw, w, d), idx)
    assert np.array_equal(pack.unpack_signs_block32(pack.pack_signs_block32(sg)), sg)
    # same bits as the row layout: bit j % 32 of row word (p, j // 32) of row r
    # equals bit β(r % 32) of block word (r // 32, p, j)
    rw = pack.pack_indices(idx, w)
    for r in (0, 1, 31, 32, 77, 95):
        for p in range(w):
            for j in (0, 17, 33, 63):
                a = (int(rw[r, p * (d // 32) + j // 32]) >> (j % 32)) & 1
                b = (int(bw[r // 32, p * d + j]) >> int(pack.block32_bit(r % 32))) & 1
                assert a == b


@pytest.mark.parametrize("w", [1, 2, 3])
def test_stage1_only_records(w):
    """Stage-1-only records hold stage 1's indices and fp32 norms and no sign rows;
    reconstructing them without the QJL term gives stage 1's n · Πᵀ c[idx].  With centroids
    at the cell means, the error is orthogonal to the reconstruction on average, so
    ⟨x, x̃⟩ / ‖x‖² = 1 − D/‖x‖² < 1: inner products through stage 1 alone are shrunk."""
    d = 64
    Pi, S, c, b, mse = _setup(d, w)
    rng = np.random.default_rng(40 + w)
    X = rng.standard_normal((300, d))
    z = quantize.quantize_mse(X, Pi, c, b)
    n, _, idx, xt = quantize.stage1(X, Pi, c, b)
    assert np.array_equal(z.idx, idx)
    assert np.array_equal(z.norm, n.astype(np.float32))
    assert z.sgn.shape == (300, 0)
    xr = quantize.reconstruct(z.idx, z.sgn, z.norm, z.rnorm, Pi, S[:0], c, qjl_stage=False)
    # the stored fp32 norm differs from the float64 one by at most half an ulp
    assert np.abs(xr - xt).max() <= 1e-7 * np.abs(xt).max()
    ip = np.sum(X * xt, axis=1) / np.sum(X * X, axis=1)
    assert abs(ip.mean() - (1.0 - d * mse)) < 5 * ip.std() / np.sqrt(len(ip)) + 1e-3
    assert ip.mean() < 1.0


@pytest.mark.parametrize("w", [1, 2, 3])
def test_tiny_workload_score_errors_match_the_closed_form_spread(w):
    """The 4096 keys and 8 queries of the tiny workload, one draw of S: the
    two-stage estimate's error e = est - ⟨q, k⟩, divided by the closed-form
    deviation √(((π/2)‖q‖²‖r‖² - ⟨q, r⟩²)/m), has mean ≈ 0 and mean square ≈ 1."""
    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED, WORKLOADS, make_kv, make_queries

    wl = WORKLOADS["tiny"]
    d = m = wl.d
    K = make_kv(wl, which=0)[0, 0].double().numpy()
    q = make_queries(wl)[0].double().numpy()
    Pi = rotation.make_rotation(d, ROTATION_SEED)
    S = qjl.make_qjl(m, d, QJL_SEED)
    c, b, _, _ = codebook.lloyd_max(d, w)
    z = quantize.quantize(K, Pi, S, c, b)
    est = q @ quantize.reconstruct(z.idx, z.sgn, z.norm, z.rnorm, Pi, S, c).T
    _, _, _, xt = quantize.stage1(K, Pi, c, b)
    R = K - xt
    qr = q @ R.T
    var = ((math.pi / 2) * np.sum(q * q, axis=1)[:, None] * np.sum(R * R, axis=1)[None, :] - qr ** 2) / m
    zs = (est - q @ K.T) / np.sqrt(var)
    assert abs(zs.mean()) < 0.03                 # 32768 errors; per-head means stay within ±0.03
    assert np.all(np.abs(zs.mean(axis=1)) < 0.06)
    assert 0.85 < np.mean(zs * zs) < 1.15
