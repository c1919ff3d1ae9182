"""Seeded random numbers drawn by the method (oracle side).

The pages fix no generator for the rotation Π or the JL matrix S.  Both sides
of this project therefore implement, each in its own code, one counter-based
generator from its published definition:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the i-th output (i = 0, 1, ...) of stream
  ``seed`` is mix64(seed + (i + 1) * 0x9E3779B97F4A7C15) (mod 2^64), with
  mix64(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31.
* uniform in (0, 1): ((z >> 11) + 0.5) * 2^-53.
* Box-Muller (Box & Muller 1958): uniforms (u1, u2) from outputs 2k, 2k+1
  give the normals sqrt(-2 ln u1) cos(2π u2) and sqrt(-2 ln u1) sin(2π u2),
  stored at positions 2k and 2k+1 of a row-major fill.

Parity: pinned by the published SplitMix64 test vector for seed 1234567 (see
tests/test_oracle_prng_rotation.py) and by moment / KS checks of the normals.
"""

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 stream ``seed`` (uint64)."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniforms(seed: int, count: int) -> np.ndarray:
    """``count`` uniforms in (0, 1) from stream ``seed`` (float64)."""
    z = splitmix64(seed, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(seed: int, count: int) -> np.ndarray:
    """``count`` standard normals by Box-Muller, pairs filled in order."""
    npairs = (count + 1) // 2
    u = uniforms(seed, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:count]


def gaussian_matrix(seed: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols matrix of iid N(0, 1), row-major fill from stream ``seed``."""
    return normals(seed, rows * cols).reshape(rows, cols)
