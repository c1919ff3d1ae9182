"""Bit packing of the stored record (oracle side).

[video] (fused-operator remarks): several small codes are packed into one
32-bit word so that the GPU reads whole words and decodes them in registers.
The pages fix no bit order.  The reading taken here packs bit-planes:

* index block, w·d/32 words per vector, plane-major: word p·(d/32) + k holds
  bit p (p = 0 is the least significant bit) of idx[32k + i] at bit i,
  i = 0..31.
* sign block, m/32 words per vector: word k holds σ[32k + i] at bit i, with
  bit value 1 <-> σ = +1.

So every stored word carries 32 consecutive coordinates of one bit-plane.

A second arrangement of the same bits serves caches that are contracted over
tokens (the value side of attention): rows are grouped in blocks of 32, and
block k holds, for plane p and coordinate j, one word whose bit
β(t) = t//2 + 16·(t mod 2) is bit p of idx[32k + t, j] (even rows in the low
half-word, odd rows in the high half); sign word j of block k likewise holds
σ[32k + t, j] at bit β(t).  Words are ordered [block][plane][coordinate] for
indices and [block][coordinate] for signs.

Parity: pinned by hand-computed words for fixed patterns and by round trips.
"""

import numpy as np

_SHIFTS = np.arange(32, dtype=np.uint64)


def _bits_to_words(bits: np.ndarray) -> np.ndarray:
    """bits [..., n] in {0, 1} with n % 32 == 0 -> uint32 words [..., n/32]."""
    n = bits.shape[-1]
    if n % 32:
        raise ValueError("bit count must be a multiple of 32")
    b = bits.astype(np.uint64).reshape(bits.shape[:-1] + (n // 32, 32))
    return np.sum(b << _SHIFTS, axis=-1).astype(np.uint32)


def _words_to_bits(words: np.ndarray) -> np.ndarray:
    w = words.astype(np.uint64)[..., None]
    b = (w >> _SHIFTS) & np.uint64(1)
    return b.reshape(words.shape[:-1] + (words.shape[-1] * 32,)).astype(np.int64)


def pack_indices(idx: np.ndarray, w: int) -> np.ndarray:
    """idx [N, d] ints in [0, 2^w) -> uint32 [N, w*d/32] (plane-major)."""
    idx = np.asarray(idx, dtype=np.int64)
    planes = [_bits_to_words((idx >> p) & 1) for p in range(w)]
    return np.concatenate(planes, axis=-1)


def unpack_indices(words: np.ndarray, w: int, d: int) -> np.ndarray:
    nw = d // 32
    idx = np.zeros(words.shape[:-1] + (d,), dtype=np.int64)
    for p in range(w):
        idx |= _words_to_bits(words[..., p * nw:(p + 1) * nw]) << p
    return idx


def pack_signs(sgn: np.ndarray) -> np.ndarray:
    """sgn [N, m] bool (True <-> +1) -> uint32 [N, m/32]."""
    return _bits_to_words(np.asarray(sgn).astype(np.int64))


def unpack_signs(words: np.ndarray) -> np.ndarray:
    return _words_to_bits(words).astype(bool)


# ---- 32-row blocks, one coordinate per word ------------------------------------

def block32_bit(t):
    """Bit position of row t (0..31) of a block: even rows low half, odd rows high half."""
    t = np.asarray(t)
    return t // 2 + 16 * (t % 2)


def _rows_to_block_words(bits: np.ndarray) -> np.ndarray:
    """bits [N, n] in {0, 1}, N % 32 == 0 -> uint32 [N/32, n] (bit β(t) of word [k, j] = bits[32k+t, j])."""
    N, n = bits.shape
    if N % 32:
        raise ValueError("row count must be a multiple of 32")
    b = bits.astype(np.uint64).reshape(N // 32, 32, n)
    shifts = block32_bit(np.arange(32)).astype(np.uint64)[None, :, None]
    return np.sum(b << shifts, axis=1).astype(np.uint32)


def _block_words_to_rows(words: np.ndarray) -> np.ndarray:
    nb, n = words.shape
    shifts = block32_bit(np.arange(32)).astype(np.uint64)[None, :, None]
    b = (words.astype(np.uint64)[:, None, :] >> shifts) & np.uint64(1)
    return b.reshape(nb * 32, n).astype(np.int64)


def pack_indices_block32(idx: np.ndarray, w: int) -> np.ndarray:
    """idx [N, d] (N % 32 == 0) -> uint32 [N/32, w*d]: words [block][plane][coordinate]."""
    idx = np.asarray(idx, dtype=np.int64)
    planes = [_rows_to_block_words((idx >> p) & 1) for p in range(w)]
    return np.concatenate(planes, axis=-1)


def unpack_indices_block32(words: np.ndarray, w: int, d: int) -> np.ndarray:
    idx = None
    for p in range(w):
        plane = _block_words_to_rows(words[:, p * d:(p + 1) * d]) << p
        idx = plane if idx is None else idx | plane
    return idx


def pack_signs_block32(sgn: np.ndarray) -> np.ndarray:
    """sgn [N, m] bool (True <-> +1), N % 32 == 0 -> uint32 [N/32, m]."""
    return _rows_to_block_words(np.asarray(sgn).astype(np.int64))


def unpack_signs_block32(words: np.ndarray) -> np.ndarray:
    return _block_words_to_rows(words).astype(bool)
