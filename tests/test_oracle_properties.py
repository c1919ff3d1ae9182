"""Property tests of the oracle's packing and bucketing over generated shapes (no GPU).

Each property holds for every input the method admits, so hypothesis draws the
shapes and values (derandomized: the same examples every run).
"""

import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

from oracle import codebook, pack, quantize

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True)


@SETTINGS
@given(w=st.integers(1, 3), words=st.integers(1, 8), n=st.integers(1, 40), seed=st.integers(0, 2 ** 31))
def test_row_packing_round_trips(w, words, n, seed):
    d = 32 * words
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, 1 << w, size=(n, d))
    sgn = rng.random((n, d)) < 0.5
    packed = pack.pack_indices(idx, w)
    assert packed.dtype == np.uint32 and packed.shape == (n, w * d // 32)
    assert np.array_equal(pack.unpack_indices(packed, w, d), idx)
    assert np.array_equal(pack.unpack_signs(pack.pack_signs(sgn)), sgn)


@SETTINGS
@given(w=st.integers(1, 3), words=st.integers(1, 4), blocks=st.integers(1, 4), seed=st.integers(0, 2 ** 31))
def test_block_packing_holds_the_row_bits(w, words, blocks, seed):
    """Bit p of idx[r][j] sits at bit β(r mod 32) of block word p·d + j, and nowhere else."""
    d, n = 32 * words, 32 * blocks
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, 1 << w, size=(n, d))
    words_b = pack.pack_indices_block32(idx, w)
    assert words_b.shape == (blocks, w * d)
    assert np.array_equal(pack.unpack_indices_block32(words_b, w, d), idx)
    r, j, p = rng.integers(0, n), rng.integers(0, d), rng.integers(0, w)
    bit = (int(words_b[r // 32, p * d + j]) >> int(pack.block32_bit(r % 32))) & 1
    assert bit == (idx[r, j] >> p) & 1
    # the 32 bit positions of a block word are a permutation of the block's rows
    assert sorted(int(pack.block32_bit(t)) for t in range(32)) == list(range(32))


@SETTINGS
@given(d=st.sampled_from([8, 16, 32, 128]), w=st.integers(1, 3), seed=st.integers(0, 2 ** 31))
def test_bucketize_picks_the_nearest_centroid(d, w, seed):
    c, b, _, _ = codebook.lloyd_max(d, w)
    rng = np.random.default_rng(seed)
    u = rng.uniform(-1.0, 1.0, size=500) * rng.choice([1.0, 0.2, 0.05])
    idx = quantize.bucketize(u, b)
    dist = np.abs(u[:, None] - c[None, :])
    best = dist.min(axis=1)
    # the chosen centroid is a nearest one (ties only on a boundary, where either is nearest)
    assert np.all(dist[np.arange(len(u)), idx] <= best + 1e-15)
    # and the cells are ordered: a larger coordinate never gets a lower cell
    order = np.argsort(u, kind="stable")
    assert np.all(np.diff(idx[order]) >= 0)


@SETTINGS
@given(d=st.sampled_from([16, 32, 64]), w=st.integers(1, 3), seed=st.integers(0, 2 ** 31),
       scale=st.floats(1e-3, 1e3))
def test_quantizer_is_scale_equivariant(d, w, seed, scale):
    """x and s·x (s > 0) get the same indices and signs; the norms scale by s."""
    from oracle import qjl, rotation

    Pi = rotation.make_rotation(d, 5)
    S = qjl.make_qjl(d, d, 6)
    c, b, _, _ = codebook.lloyd_max(d, w)
    X = np.random.default_rng(seed).standard_normal((8, d))
    z1 = quantize.quantize(X, Pi, S, c, b)
    z2 = quantize.quantize(scale * X, Pi, S, c, b)
    # rounding can move a coordinate that lies on a boundary; compare the clear ones
    clear = np.abs(z1.u[..., None] - b).min(axis=-1) > 1e-12
    assert np.array_equal(z1.idx[clear], z2.idx[clear])
    assert np.allclose(z2.rnorm64, scale * z1.rnorm64, rtol=1e-10, atol=0)
    clear_s = (np.abs(z1.p) > 1e-9 * np.abs(z1.p).max()) & np.all(clear, axis=1)[:, None]
    assert np.array_equal(z1.sgn[clear_s], z2.sgn[clear_s])
