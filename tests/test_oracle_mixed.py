"""Pins for the oracle's outlier-channel split precision (no GPU).

Reading ("TurboQuant压缩效果" transcripts, 2.5 / 3.5 bits): the channels of a
head split into outliers (b + 1 total bits) and the rest (b bits), each side
quantized by its own TurboQuant instance; scores add, reconstructions sit at
their own channels.
"""

import numpy as np
import pytest

from oracle import codebook, mixed, quantize


def _tables(d=64, n_o=32, bits=2, seed=5):
    rng = np.random.default_rng(seed)
    perm = np.sort(rng.permutation(d)[:n_o]).astype(np.int64)
    rest = np.array(sorted(set(range(d)) - set(perm.tolist())), dtype=np.int64)
    perm = np.concatenate([perm, rest])
    return mixed.make_tables(perm, n_o, bits, 101, 102, 103, 104)


def test_bit_accounting_matches_the_page_labels():
    """2.5 and 3.5 bits per coordinate: regular channels at 2 or 3 bits, half the
    128 channels one bit higher; the four fp32 norms add one bit at d = 128."""
    assert mixed.bits_per_coordinate(128, 64, 2) == 2.5
    assert mixed.bits_per_coordinate(128, 64, 3) == 3.5
    assert mixed.bits_per_coordinate(128, 64, 2, with_norms=True) == 3.5
    assert mixed.bits_per_coordinate(128, 32, 2) == 2.25


def test_choose_outliers_finds_planted_channels():
    rng = np.random.default_rng(1)
    d = 128
    X = rng.standard_normal((4096, d))
    planted = np.array([3, 40, 77, 120])
    X[:, planted] *= 20.0
    perm = mixed.choose_outliers(X, 4)
    assert np.array_equal(perm[:4], planted)
    assert np.array_equal(np.sort(perm), np.arange(d))
    perm32 = mixed.choose_outliers(X, 32)
    assert set(planted.tolist()) <= set(perm32[:32].tolist())
    assert np.all(np.diff(perm32[:32]) > 0) and np.all(np.diff(perm32[32:]) > 0)


def test_codeword_rays_of_both_instances_keep_their_cells_and_channels():
    """x whose outlier part is t_O·Π_Oᵀc_O[i_O] and regular part t_R·Π_Rᵀc_R[i_R]:
    each side keeps its planted indices and norm, and the stage-1 reconstruction
    puts ‖x_part‖·Π_partᵀ c[i_part] back at exactly that side's channels."""
    t = _tables()
    rng = np.random.default_rng(2)

    def ray(Pi, c, b, dim, n):
        idx = rng.integers(0, len(c), size=(n, dim))
        cn = np.linalg.norm(c[idx], axis=1)
        v = c[idx] / cn[:, None]
        lo = np.concatenate([[-np.inf], b])[idx]
        hi = np.concatenate([b, [np.inf]])[idx]
        keep = np.all((v > lo + 1e-9) & (v < hi - 1e-9), axis=1)
        return idx[keep], cn[keep]

    iO, cnO = ray(t.Pi_O, t.c_O, t.b_O, t.n_o, 400)
    iR, cnR = ray(t.Pi_R, t.c_R, t.b_R, t.perm.shape[0] - t.n_o, 400)
    n = min(len(iO), len(iR), 20)
    assert n >= 5
    iO, cnO, iR, cnR = iO[:n], cnO[:n], iR[:n], cnR[:n]
    tO, tR = 2.0 ** rng.integers(-2, 3, size=n), 2.0 ** rng.integers(-2, 3, size=n)
    X = np.zeros((n, t.perm.shape[0]))
    X[:, t.perm[:t.n_o]] = tO[:, None] * (t.c_O[iO] @ t.Pi_O)
    X[:, t.perm[t.n_o:]] = tR[:, None] * (t.c_R[iR] @ t.Pi_R)
    qO, qR = mixed.quantize_split(X, t)
    assert np.array_equal(qO.idx, iO) and np.array_equal(qR.idx, iR)
    assert np.allclose(qO.norm, tO * cnO, rtol=1e-7) and np.allclose(qR.norm, tR * cnR, rtol=1e-7)
    xt = mixed.reconstruct_split(qO, qR, t, qjl_stage=False)
    want = np.zeros_like(X)
    want[:, t.perm[:t.n_o]] = np.asarray(qO.norm, np.float64)[:, None] * (t.c_O[iO] @ t.Pi_O)
    want[:, t.perm[t.n_o:]] = np.asarray(qR.norm, np.float64)[:, None] * (t.c_R[iR] @ t.Pi_R)
    assert np.allclose(xt, want, rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3])
def test_stage1_distortion_of_each_side_is_its_own_codebook_mse(bits):
    """For isotropic Gaussian x, Π_part x_part/‖x_part‖ is uniform on its sphere, so
    E‖x_part - x̃_part‖²/‖x_part‖² = d_part · MSE(d_part, w_part): outliers at
    w = bits, the rest at w = bits - 1."""
    t = _tables(bits=bits)
    rng = np.random.default_rng(3 + bits)
    X = rng.standard_normal((20000, t.perm.shape[0]))
    qO, qR = mixed.quantize_split(X, t)
    xt = mixed.reconstruct_split(qO, qR, t, qjl_stage=False)
    for ch, dim, w in ((t.perm[:t.n_o], t.n_o, bits), (t.perm[t.n_o:], t.perm.shape[0] - t.n_o, bits - 1)):
        err = np.sum((X[:, ch] - xt[:, ch]) ** 2, axis=1) / np.sum(X[:, ch] ** 2, axis=1)
        _, _, mse, _ = codebook.lloyd_max(dim, w)
        assert abs(err.mean() / (dim * mse) - 1.0) < 0.03, (dim, w, err.mean(), dim * mse)


def test_split_score_is_unbiased_over_qjl_draws():
    """With the rotations fixed, the mean of the split estimator over 10^4
    independent pairs of QJL matrices is within 3 standard errors of ⟨q, x⟩."""
    t0 = _tables(d=64, n_o=32, bits=2, seed=9)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 64))
    q = rng.standard_normal(64)
    draws = 10000
    est = np.empty(draws)
    for i in range(draws):
        t = mixed.SplitTables(perm=t0.perm, n_o=t0.n_o, Pi_O=t0.Pi_O, S_O=rng.standard_normal((32, 32)), c_O=t0.c_O,
                              b_O=t0.b_O, Pi_R=t0.Pi_R, S_R=rng.standard_normal((32, 32)), c_R=t0.c_R, b_R=t0.b_R)
        qO, qR = mixed.quantize_split(x, t)
        est[i] = mixed.score_split(q, qO, qR, t)[0]
    truth = float(x[0] @ q)
    se = est.std(ddof=1) / np.sqrt(draws)
    assert abs(est.mean() - truth) < 3 * se, (est.mean(), truth, se)


def test_single_token_attention_returns_that_value():
    """ctx_len = 1: softmax weight 1, the output is the reconstruction of value 0."""
    t = _tables(d=64, n_o=32, bits=2)
    rng = np.random.default_rng(6)
    B, Hkv, T, d = 1, 1, 3, 64
    K = rng.standard_normal((B * Hkv * T, d))
    V = rng.standard_normal((B * Hkv * T, d))
    kO, kR = mixed.quantize_split(K, t)
    vO, vR = mixed.quantize_split(V, t)

    def rec(qq, dim):
        return {"idx": qq.idx.reshape(B, Hkv, T, dim), "sgn": qq.sgn.reshape(B, Hkv, T, dim),
                "norm": qq.norm.reshape(B, Hkv, T), "rnorm": qq.rnorm.reshape(B, Hkv, T)}

    q = rng.standard_normal((B, 2, d))
    out, _ = mixed.decode_attention_split(q, rec(kO, 32), rec(kR, 32), rec(vO, 32), rec(vR, 32), [1], t)
    v0 = mixed.reconstruct_split(vO, vR, t)[0]
    assert np.allclose(out[0, 0], v0, rtol=1e-12, atol=1e-12)
    assert np.allclose(out[0, 1], v0, rtol=1e-12, atol=1e-12)
    # the split score of key 0 for head 0 is what the attention saw
    s = mixed.score_split(q[0, 0], kO, kR, t)
    k0 = mixed.reconstruct_split(kO, kR, t)
    assert np.allclose(s, k0 @ q[0, 0], rtol=1e-10, atol=1e-10)
    # and it reduces to the single-instance estimator on each side
    sO = quantize.reconstruct(kO.idx, kO.sgn, kO.norm, kO.rnorm, t.Pi_O, t.S_O, t.c_O) @ q[0, 0][t.perm[:32]]
    sR = quantize.reconstruct(kR.idx, kR.sgn, kR.norm, kR.rnorm, t.Pi_R, t.S_R, t.c_R) @ q[0, 0][t.perm[32:]]
    assert np.allclose(s, sO + sR, rtol=1e-10, atol=1e-10)
