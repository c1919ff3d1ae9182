"""Planted mistakes in the oracle must fail its pins.

Each case swaps one oracle function (or constant), on the CPU and only for the
length of one test, for a version carrying one plausible slip -- a dropped
factor, a transposed operand, a wrong index, sign, tie rule or bit order --
and runs the pin meant to catch that slip, which has to fail.  The oracle's
files are never edited; the swap is a pytest monkeypatch.
"""

import math
from dataclasses import dataclass
from typing import Callable

import numpy as np
import pytest

from oracle import codebook, decode, pack, prng, qjl, quantize, rotation, search

import test_oracle_codebook as t_cb
import test_oracle_decode_search as t_ds
import test_oracle_prng_rotation as t_pr
import test_oracle_quantize as t_q


@dataclass
class Mutant:
    name: str
    target: object           # module holding the name
    attr: str                # name swapped
    make: Callable           # original -> replacement
    pin: Callable            # a pin that must now fail


# ---- replacements that need more than a wrapper around the original --------

def _normals_cos_twice(seed, count):
    """Box-Muller that takes the cosine for both members of a pair."""
    npairs = (count + 1) // 2
    u = prng.uniforms(seed, 2 * npairs)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = 2.0 * np.pi * u[1::2]
    out = np.empty(2 * npairs)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.cos(t)
    return out[:count]


def _gamma_ratio_step_slip(d):
    """Γ(d/2)/Γ((d-1)/2) by the recurrence with the step k/(k+1) for k/(k-1)."""
    r = math.sqrt(math.pi) / 2.0 if d % 2 == 1 else 2.0 / math.sqrt(math.pi)
    for k in range(3 if d % 2 == 1 else 4, d, 2):
        r *= k / (k + 1.0)
    return r


def _half_moment_exponent_slip(a, b, d):
    """∫ x f_d with the antiderivative's exponent left at (d-3)/2."""
    e = (d - 3) / 2.0
    return codebook.density_const(d) * ((1.0 - a * a) ** e - (1.0 - min(b, 1.0) ** 2) ** e) / (2.0 * e)


def _half_mass_unsquared(a, b, d):
    """P(a ≤ X ≤ b) through the incomplete beta at b and a instead of b² and a²."""
    from scipy import special

    bb = (d - 1) / 2.0
    if b >= 1.0:
        return 0.5 * special.betaincc(0.5, bb, a)
    return 0.5 * (special.betainc(0.5, bb, b) - special.betainc(0.5, bb, a))


def _density_exponent_slip(x, d):
    x = np.asarray(x, dtype=np.float64)
    return codebook.density_const(d) * np.power(np.clip(1.0 - x * x, 0.0, None), (d - 1) / 2.0)


def _stage1_transposed(X, Pi, centroids, bounds):
    """Stage 1 rotating by Πᵀ (x @ Π) instead of Π."""
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=1))
    u = (X @ Pi) / np.where(n > 0.0, n, 1.0)[:, None]
    idx = quantize.bucketize(u, bounds)
    return n, u, idx, n[:, None] * (centroids[idx] @ Pi)


def _stage1_no_norm(X, Pi, centroids, bounds):
    """Stage 1 whose reconstruction forgets the factor ‖x‖."""
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=1))
    u = (X @ Pi.T) / np.where(n > 0.0, n, 1.0)[:, None]
    idx = quantize.bucketize(u, bounds)
    return n, u, idx, centroids[idx] @ Pi


def _quantize_residual_flipped(X, Pi, S, centroids, bounds):
    """Two-stage quantizer taking the residual as x̃ - x."""
    n, u, idx, xt = quantize.stage1(X, Pi, centroids, bounds)
    r = xt - np.asarray(X, dtype=np.float64)
    p = r @ S.T
    rn = np.sqrt(np.sum(r * r, axis=1))
    return quantize.Quantized(idx=idx, sgn=p >= 0.0, norm=n.astype(np.float32), rnorm=rn.astype(np.float32),
                              u=u, p=p, rnorm64=rn)


def _signs_stored_inverted(f):
    """Two-stage quantizer storing True for σ = -1."""
    def quant(*args):
        z = f(*args)
        z.sgn = ~z.sgn
        return z
    return quant


def _rnorm_of_x(f):
    """Two-stage quantizer storing ‖x‖ where ‖r‖ belongs (the plain-QJL norm)."""
    def quant(*args):
        z = f(*args)
        z.rnorm = z.norm.copy()
        return z
    return quant


def _decode_dropping_qjl(keys):
    """Attention over records that leaves out the QJL term of the keys (or of the values)."""
    def dec(q, K_rec, V_rec, ctx_len, Pi, S, centroids, scale=None, qjl_stage=True):
        Kh = decode.reconstruct_cache(K_rec, Pi, S, centroids, qjl_stage=not keys)
        Vh = decode.reconstruct_cache(V_rec, Pi, S, centroids, qjl_stage=keys)
        return decode.attention(q, Kh, Vh, ctx_len, scale)
    return dec


def _reconstruct_with(alpha, transpose_s):
    def rec(idx, sgn, norm, rnorm, Pi, S, centroids, qjl_stage=True):
        m = S.shape[0]
        x = np.asarray(norm, dtype=np.float64)[:, None] * (centroids[idx] @ Pi)
        if qjl_stage:
            sig = np.where(sgn, 1.0, -1.0)
            proj = sig @ (S.T if transpose_s else S)
            x = x + alpha(m) * np.asarray(rnorm, dtype=np.float64)[:, None] * proj
        return x
    return rec


def _attention_interleaved_heads(q, Kh, Vh, ctx_len, scale=None):
    """Attention that maps query head g to kv head g mod Hkv."""
    B, Hq, d = q.shape
    Hkv = Kh.shape[1]
    scale = 1.0 / np.sqrt(d) if not scale else scale
    out = np.zeros((B, Hq, d))
    scores = np.full((B, Hq, Kh.shape[2]), -np.inf)
    for b in range(B):
        L = int(ctx_len[b])
        for g in range(Hq):
            s = scale * (Kh[b, g % Hkv, :L] @ q[b, g])
            scores[b, g, :L] = s
            e = np.exp(s - s.max())
            out[b, g] = (e / e.sum()) @ Vh[b, g % Hkv, :L]
    return out, scores


def _topk_reversed_ties(Q, rec, Pi, S, centroids, k, qjl_stage=True):
    """Top-k taken from the end of an ascending sort, which puts equal scores highest index first."""
    sc = search.scores(Q, rec, Pi, S, centroids, qjl_stage=qjl_stage)
    order = np.argsort(sc, axis=1, kind="stable")[:, ::-1][:, :k]
    return order, np.take_along_axis(sc, order, axis=1)


MUTANTS = [
    # generator and rotation
    Mutant("splitmix_counter_from_zero", prng, "splitmix64",
           lambda f: (lambda seed, count, start=0: f(seed, count, start + 1)),
           t_pr.test_splitmix64_published_sequence),
    Mutant("box_muller_cosine_twice", prng, "normals", lambda f: _normals_cos_twice,
           t_pr.test_box_muller_normals_are_standard_normal),
    Mutant("rotation_without_qr_sign_fix", rotation, "make_rotation",
           lambda f: (lambda d, seed: np.linalg.qr(prng.gaussian_matrix(seed, d, d))[0]),
           lambda: t_pr.test_rotation_is_the_positive_diagonal_qr_factor(8)),
    Mutant("rotation_transposed", rotation, "make_rotation", lambda f: (lambda d, seed: f(d, seed).T),
           lambda: t_pr.test_rotation_is_the_positive_diagonal_qr_factor(128)),
    # codebook
    Mutant("gamma_ratio_recurrence_step", codebook, "gamma_half_ratio", lambda f: _gamma_ratio_step_slip,
           lambda: t_cb.test_one_bit_closed_form(128)),
    Mutant("conditional_moment_exponent", codebook, "_half_moment", lambda f: _half_moment_exponent_slip,
           lambda: t_cb.test_one_bit_closed_form(8)),
    Mutant("cell_mass_unsquared_bounds", codebook, "_half_mass", lambda f: _half_mass_unsquared,
           lambda: t_cb.test_centroids_are_conditional_means_by_quadrature(8, 2)),
    Mutant("density_exponent", codebook, "density", lambda f: _density_exponent_slip,
           lambda: t_cb.test_centroids_are_conditional_means_by_quadrature(128, 2)),
    # quantizer
    Mutant("bucketize_magnitude_only", quantize, "bucketize", lambda f: (lambda u, b: f(np.abs(u), b)),
           lambda: t_q.test_bucketize_is_brute_force_nearest_codeword(2)),
    Mutant("bucketize_ties_to_upper_cell", quantize, "bucketize",
           lambda f: (lambda u, b: np.searchsorted(b, u, side="right").astype(np.int64)),
           t_q.test_zero_vector_rule),
    Mutant("stage1_rotates_by_transpose", quantize, "stage1", lambda f: _stage1_transposed,
           lambda: t_q.test_vectors_on_a_codeword_ray(2)),
    Mutant("stage1_reconstruction_without_norm", quantize, "stage1", lambda f: _stage1_no_norm,
           lambda: t_q.test_vectors_on_a_codeword_ray(3)),
    Mutant("residual_sign_flipped", quantize, "quantize", lambda f: _quantize_residual_flipped,
           t_q.test_two_stage_score_is_unbiased_over_S),
    Mutant("stored_sign_convention_inverted", quantize, "quantize", _signs_stored_inverted,
           t_q.test_two_stage_score_is_unbiased_over_S),
    Mutant("residual_norm_replaced_by_vector_norm", quantize, "quantize", _rnorm_of_x,
           lambda: t_q.test_tiny_workload_score_errors_match_the_closed_form_spread(2)),
    Mutant("qjl_scale_without_sqrt_pi_over_2", qjl, "qjl_alpha", lambda f: (lambda m: 1.0 / m),
           t_q.test_qjl_estimator_unbiased_with_closed_form_variance),
    Mutant("qjl_signs_of_transposed_s", qjl, "signs", lambda f: (lambda S, r: f(S.T, r)),
           t_q.test_qjl_estimator_unbiased_with_closed_form_variance),
    Mutant("reconstruct_scale_one_over_m", quantize, "reconstruct",
           lambda f: _reconstruct_with(lambda m: 1.0 / m, False),
           t_q.test_two_stage_score_is_unbiased_over_S),
    Mutant("reconstruct_transposed_s", quantize, "reconstruct",
           lambda f: _reconstruct_with(qjl.qjl_alpha, True),
           t_q.test_reconstruct_inner_product_is_the_estimator),
    # packing
    Mutant("bits_msb_first", pack, "_SHIFTS", lambda v: v[::-1].copy(), t_q.test_pack_hand_patterns),
    Mutant("block32_rows_in_order", pack, "block32_bit", lambda f: (lambda t: np.asarray(t)),
           t_q.test_pack_block32_hand_patterns),
    # attention and search
    Mutant("attention_scale_one_over_d", decode, "attention",
           lambda f: (lambda q, K, V, ctx, scale=None: f(q, K, V, ctx, scale or 1.0 / q.shape[-1])),
           t_ds.test_exact_codewords_reduce_to_library_attention),
    Mutant("attention_heads_interleaved", decode, "attention", lambda f: _attention_interleaved_heads,
           t_ds.test_gqa_consecutive_grouping),
    Mutant("attention_ignores_context_length", decode, "attention",
           lambda f: (lambda q, K, V, ctx, scale=None: f(q, K, V, np.full(len(ctx), K.shape[2]), scale)),
           t_ds.test_zero_query_is_mean_of_values),
    Mutant("keys_drop_qjl_term", decode, "decode_attention", lambda f: _decode_dropping_qjl(keys=True),
           t_ds.test_decode_scores_are_the_two_stage_estimator),
    Mutant("values_drop_qjl_term", decode, "decode_attention", lambda f: _decode_dropping_qjl(keys=False),
           t_ds.test_context_one_output_is_the_value_estimator),
    Mutant("search_drops_qjl_term", search, "reconstruct",
           lambda f: (lambda *a, qjl_stage=True: f(*a, qjl_stage=False)),
           t_ds.test_search_scores_are_the_two_stage_estimator),
    Mutant("search_ties_to_higher_index", search, "topk", lambda f: _topk_reversed_ties,
           t_ds.test_search_ties_go_to_lower_index),
]


def test_every_oracle_module_has_a_mutant():
    hit = {m.target.__name__ for m in MUTANTS}
    assert hit == {f"oracle.{n}" for n in ("prng", "rotation", "codebook", "quantize", "qjl", "pack", "decode",
                                           "search")}


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.name for m in MUTANTS])
def test_pin_fails_on_planted_mistake(mutant, monkeypatch):
    mutant.pin()  # the pin passes on the oracle as it stands
    monkeypatch.setattr(mutant.target, mutant.attr, mutant.make(getattr(mutant.target, mutant.attr)))
    # a failed assertion, or arithmetic that breaks down on the wrong values
    with pytest.raises((AssertionError, ArithmeticError)):
        mutant.pin()
