"""Pins for the oracle's attention and search over stored records (no GPU)."""

import numpy as np
import torch

from oracle import codebook, decode, qjl, quantize, rotation, search


def _cache(B, H, T, d, m, w, seed, exact=False):
    Pi = rotation.make_rotation(d, 100 + seed)
    S = qjl.make_qjl(m, d, 200 + seed)
    c, b, _, _ = codebook.lloyd_max(d, w)
    rng = np.random.default_rng(seed)
    if exact:
        # records with a zero residual norm reconstruct to norm · Πᵀ c[idx] exactly
        n = B * H * T
        idx = rng.integers(0, 1 << w, size=(n, d))
        nrm = 2.0 ** rng.integers(-2, 3, size=n)
        X = nrm[:, None] * (c[idx] @ Pi)
        rec = {"idx": idx, "sgn": rng.integers(0, 2, size=(n, m)).astype(bool),
               "norm": nrm.astype(np.float32), "rnorm": np.zeros(n, np.float32)}
    else:
        X = rng.standard_normal((B * H * T, d)) * (1 + 5 * (rng.random(d) < 0.05))
        z = quantize.quantize(X, Pi, S, c, b)
        rec = {"idx": z.idx, "sgn": z.sgn, "norm": z.norm, "rnorm": z.rnorm}
    rec = {k: v.reshape((B, H, T) + v.shape[1:]) for k, v in rec.items()}
    return X.reshape(B, H, T, d), rec, Pi, S, c


def test_exact_codewords_reduce_to_library_attention():
    B, Hq, Hkv, T, d, w = 2, 4, 2, 40, 32, 2
    K, Krec, Pi, S, c = _cache(B, Hkv, T, d, d, w, 1, exact=True)
    V, Vrec, _, _, _ = _cache(B, Hkv, T, d, d, w, 1, exact=True)
    V = V[:, :, ::-1].copy()  # distinct values, same codeword construction
    Vrec = {k: v[:, :, ::-1].copy() for k, v in Vrec.items()}
    q = np.random.default_rng(3).standard_normal((B, Hq, d))
    ctx = np.array([T, 17])
    out, _ = decode.decode_attention(q, Krec, Vrec, ctx, Pi, S, c)
    for bi in range(B):
        L = ctx[bi]
        qt = torch.tensor(q[bi:bi + 1], dtype=torch.float64)            # [1, Hq, d]
        kt = torch.tensor(K[bi:bi + 1, :, :L], dtype=torch.float64).repeat_interleave(Hq // Hkv, dim=1)
        vt = torch.tensor(V[bi:bi + 1, :, :L], dtype=torch.float64).repeat_interleave(Hq // Hkv, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(qt[:, :, None], kt, vt)[:, :, 0]
        assert np.abs(out[bi] - ref[0].numpy()).max() < 1e-12


def _estimate(rec, at, y, Pi, S, c):
    """The two-stage estimate of ⟨x, y⟩ for the record at index ``at``, piece by
    piece: ‖x‖ ⟨Π y, c[idx]⟩ + √(π/2)/m ‖r‖ ⟨S y, σ⟩."""
    stage1 = float(rec["norm"][at]) * float(c[rec["idx"][at]] @ (Pi @ y))
    sig = np.where(rec["sgn"][at], 1.0, -1.0)
    return stage1 + qjl.estimate(S, y, float(rec["rnorm"][at]), sig)


def test_decode_scores_are_the_two_stage_estimator():
    """Every logit is the key's two-stage inner-product estimate times 1/√d."""
    B, Hq, Hkv, T, d, w = 2, 4, 2, 12, 32, 2
    _, Krec, Pi, S, c = _cache(B, Hkv, T, d, d, w, 14)
    _, Vrec, _, _, _ = _cache(B, Hkv, T, d, d, w, 15)
    q = np.random.default_rng(7).standard_normal((B, Hq, d))
    ctx = np.array([T, 5])
    _, sc = decode.decode_attention(q, Krec, Vrec, ctx, Pi, S, c)
    for bi in range(B):
        for g in range(Hq):
            h = g // (Hq // Hkv)
            for t in range(T):
                if t >= ctx[bi]:
                    assert sc[bi, g, t] == -np.inf
                    continue
                est = _estimate(Krec, (bi, h, t), q[bi, g], Pi, S, c)
                assert abs(sc[bi, g, t] - est / np.sqrt(d)) < 1e-12 * (1 + abs(est))


def test_context_one_output_is_the_value_estimator():
    """With one token the output is that value's reconstruction: ⟨o, y⟩ is the
    two-stage estimate of ⟨v, y⟩ for any y."""
    B, H, T, d, w = 1, 1, 4, 32, 3
    _, Krec, Pi, S, c = _cache(B, H, T, d, d, w, 16)
    _, Vrec, _, _, _ = _cache(B, H, T, d, d, w, 17)
    rng = np.random.default_rng(8)
    out, _ = decode.decode_attention(rng.standard_normal((B, 3, d)), Krec, Vrec, np.array([1]), Pi, S, c)
    for y in rng.standard_normal((4, d)):
        est = _estimate(Vrec, (0, 0, 0), y, Pi, S, c)
        for g in range(3):
            assert abs(out[0, g] @ y - est) < 1e-12 * (1 + abs(est))


def test_context_one_returns_reconstructed_value():
    B, H, T, d, w = 1, 1, 8, 32, 3
    _, Krec, Pi, S, c = _cache(B, H, T, d, d, w, 4)
    _, Vrec, _, _, _ = _cache(B, H, T, d, d, w, 5)
    q = np.random.default_rng(0).standard_normal((B, 2, d))
    out, _ = decode.decode_attention(q, Krec, Vrec, np.array([1]), Pi, S, c)
    vh = decode.reconstruct_cache(Vrec, Pi, S, c)
    assert np.abs(out[0] - vh[0, 0, 0][None, :]).max() < 1e-13


def test_zero_query_is_mean_of_values():
    B, H, T, d, w = 1, 1, 30, 32, 2
    _, Krec, Pi, S, c = _cache(B, H, T, d, d, w, 6)
    _, Vrec, _, _, _ = _cache(B, H, T, d, d, w, 7)
    out, _ = decode.decode_attention(np.zeros((1, 1, d)), Krec, Vrec, np.array([21]), Pi, S, c)
    vh = decode.reconstruct_cache(Vrec, Pi, S, c)
    assert np.abs(out[0, 0] - vh[0, 0, :21].mean(axis=0)).max() < 1e-13


def test_token_permutation_invariance():
    B, H, T, d, w = 1, 2, 25, 32, 2
    _, Krec, Pi, S, c = _cache(B, H, T, d, d, w, 8)
    _, Vrec, _, _, _ = _cache(B, H, T, d, d, w, 9)
    q = np.random.default_rng(2).standard_normal((B, 4, d))
    ctx = np.array([T])
    out, _ = decode.decode_attention(q, Krec, Vrec, ctx, Pi, S, c)
    perm = np.random.default_rng(3).permutation(T)
    Kp = {k: v[:, :, perm] for k, v in Krec.items()}
    Vp = {k: v[:, :, perm] for k, v in Vrec.items()}
    outp, _ = decode.decode_attention(q, Kp, Vp, ctx, Pi, S, c)
    assert np.abs(out - outp).max() < 1e-12


def test_gqa_consecutive_grouping():
    B, Hkv, T, d, w = 1, 2, 10, 32, 2
    _, Krec, Pi, S, c = _cache(B, Hkv, T, d, d, w, 10)
    _, Vrec, _, _, _ = _cache(B, Hkv, T, d, d, w, 11)
    # make every value of kv head 1 the same record -> its query heads return it
    for k in Vrec:
        Vrec[k][:, 1] = Vrec[k][:, 1, :1]
    q = np.random.default_rng(4).standard_normal((B, 4, d))
    out, _ = decode.decode_attention(q, Krec, Vrec, np.array([T]), Pi, S, c)
    vh = decode.reconstruct_cache(Vrec, Pi, S, c)
    assert np.abs(out[0, 2:] - vh[0, 1, 0]).max() < 1e-12
    assert np.abs(out[0, 0] - vh[0, 1, 0]).max() > 1e-3


def test_search_exact_codewords_is_brute_force_mips():
    N, d, w = 300, 32, 3
    X, rec, Pi, S, c = _cache(1, 1, N, d, d, w, 12, exact=True)
    X = X.reshape(N, d)
    rec = {k: v.reshape((N,) + v.shape[3:]) for k, v in rec.items()}
    Q = np.random.default_rng(5).standard_normal((6, d))
    idx, sc = search.topk(Q, rec, Pi, S, c, 10)
    for i in range(6):
        ref = np.argsort(-(X @ Q[i]))[:10]
        assert np.array_equal(idx[i], ref)
        assert np.allclose(sc[i], (X @ Q[i])[ref], rtol=1e-12, atol=1e-12)


def test_search_scores_are_the_two_stage_estimator():
    N, d, w = 40, 32, 3
    _, rec, Pi, S, c = _cache(1, 1, N, d, d, w, 18)
    rec = {k: v.reshape((N,) + v.shape[3:]) for k, v in rec.items()}
    Q = np.random.default_rng(9).standard_normal((3, d))
    sc = search.scores(Q, rec, Pi, S, c)
    for i in range(3):
        for j in range(N):
            est = _estimate(rec, j, Q[i], Pi, S, c)
            assert abs(sc[i, j] - est) < 1e-12 * (1 + abs(est))


def test_search_ties_go_to_lower_index():
    N, d, w = 20, 32, 2
    _, rec, Pi, S, c = _cache(1, 1, N, d, d, w, 13)
    rec = {k: v.reshape((N,) + v.shape[3:]) for k, v in rec.items()}
    for k in rec:
        rec[k][7] = rec[k][3]
        rec[k][15] = rec[k][3]
    Q = np.random.default_rng(6).standard_normal((40, d))
    idx, _ = search.topk(Q, rec, Pi, S, c, N)
    for row in idx:
        pos = [list(row).index(i) for i in (3, 7, 15)]
        assert pos == sorted(pos)
