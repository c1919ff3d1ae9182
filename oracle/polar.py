"""PolarQuant's recursive polar stage, an alternative stage 1 (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "TurboQuant 与 AI 效率革命" §二 "突破：极坐标" (recursive transform to
one radius and d - 1 angles, the angle law and its mean π/4, a fixed codebook
with no normalisation constants); the csdn explainer's polar-coordinate
section; "TurboQuant压缩效果" (four bits for the first level, two for later
ones).

Transform of a rotated vector u ∈ R^d, d a power of two:
  level 1:     pairs (u_2i, u_2i+1) -> radius ρ_i = √(u_2i² + u_2i+1²) and
               angle ψ_i = atan2(u_2i+1, u_2i) taken in [0, 2π);
  level ℓ ≥ 2: pairs of level ℓ-1 radii (ρ_a, ρ_b) -> radius √(ρ_a² + ρ_b²)
               and angle atan2(ρ_b, ρ_a) in [0, π/2];
  after log2(d) levels one radius (= ‖u‖) and d - 1 angles remain.

Angle laws for a Gaussian (or uniformly rotated) u: level-1 angles are
uniform on [0, 2π).  A level-ℓ angle splits two radii that each gather
k = 2^(ℓ-1) coordinates; its density is the page's

    f_k(ψ) = Γ(k) / (2^(k-2) Γ(k/2)²) · sin^(k-1)(2ψ),   0 ≤ ψ ≤ π/2,

read with the page's d as k (it is the law of ψ = arccos(1 - 2v)/2 with
v ~ Beta(k/2, k/2), so P(ψ ≤ t) = I_{sin² t}(k/2, k/2)); its mean is π/4.

Quantizer (reading): level-1 angles take b1 = 4 bits on 2^b1 equal cells of
[0, 2π) with the cell midpoints as centroids (the Lloyd-Max quantizer of a
uniform law); every later angle takes b = 2 bits on the Lloyd-Max codebook of
its f_k (float64, by quadrature; ties go to the lower cell).  Stored: the
angle indices and ‖x‖ as fp32.  Reconstruction runs the tree back from the
radius: ρ_a = R cos ψ̃, ρ_b = R sin ψ̃, ..., u_2i = ρ_i cos ψ̃_i,
u_2i+1 = ρ_i sin ψ̃_i, and x̃ = Πᵀ ũ.

As TurboQuant's first stage ("TurboQuant 与 AI 效率革命" §四: polar stage,
then the 1-bit QJL correction) the residual r = x - x̃ goes through the same
QJL stage as quantize.quantize: σ = sign(S r), ‖r‖ fp32.

Bits per vector at d = 128, b1 = 4, b = 2: 64·4 + 63·2 = 382 angle bits,
about 3 bits per coordinate, plus 32 for the radius ("TurboQuant压缩效果":
the first level at 4 bits, later levels at 2, which is why it lands near 3).

Parity: pinned by the density's normalisation and mean π/4, its CDF against
the incomplete-beta closed form, a KS test of the transform's angles of
Gaussian vectors against those laws, the exact round trip of the transform,
the Lloyd-Max optimality conditions by independent quadrature, the uniform
quantizer's Δ²/12 distortion, and exact re-quantization of vectors built
from centroids.
"""

import math
from dataclasses import dataclass

import numpy as np
from scipy import integrate, special


def levels(d: int) -> int:
    L = int(round(math.log2(d)))
    if 1 << L != d or d < 2:
        raise ValueError("d must be a power of two >= 2")
    return L


def angle_density(psi, k: int):
    """f_k(ψ) on [0, π/2] (the page's formula with d = k)."""
    psi = np.asarray(psi, dtype=np.float64)
    c = math.exp(math.lgamma(k) - (k - 2) * math.log(2.0) - 2.0 * math.lgamma(k / 2.0))
    return c * np.power(np.clip(np.sin(2.0 * psi), 0.0, None), k - 1)


def angle_cdf(t, k: int):
    """P(ψ ≤ t) = I_{sin² t}(k/2, k/2)."""
    t = np.asarray(t, dtype=np.float64)
    return special.betainc(k / 2.0, k / 2.0, np.sin(t) ** 2)


def forward(U: np.ndarray):
    """Rows of U [N, d] -> (radius [N], angles list over levels: level ℓ an [N, d/2^ℓ] array)."""
    U = np.asarray(U, dtype=np.float64)
    d = U.shape[1]
    L = levels(d)
    x, y = U[:, 0::2], U[:, 1::2]
    rho = np.sqrt(x * x + y * y)
    angles = [np.mod(np.arctan2(y, x), 2.0 * np.pi)]
    for _ in range(2, L + 1):
        a, b = rho[:, 0::2], rho[:, 1::2]
        angles.append(np.arctan2(b, a))
        rho = np.sqrt(a * a + b * b)
    return rho[:, 0], angles


def inverse(radius: np.ndarray, angles) -> np.ndarray:
    """The transform run backwards: (radius, angles by level) -> U [N, d]."""
    rho = np.asarray(radius, dtype=np.float64)[:, None]
    for ang in reversed(angles[1:]):
        nxt = np.empty((rho.shape[0], 2 * rho.shape[1]))
        nxt[:, 0::2] = rho * np.cos(ang)
        nxt[:, 1::2] = rho * np.sin(ang)
        rho = nxt
    ang = angles[0]
    U = np.empty((rho.shape[0], 2 * rho.shape[1]))
    U[:, 0::2] = rho * np.cos(ang)
    U[:, 1::2] = rho * np.sin(ang)
    return U


def uniform_codebook(bits: int):
    """Level-1 quantizer of [0, 2π): 2^bits equal cells, centroids at their midpoints."""
    n = 1 << bits
    step = 2.0 * np.pi / n
    bounds = step * np.arange(1, n)
    centroids = step * (np.arange(n) + 0.5)
    return centroids, bounds


def lloyd_max_angle(k: int, bits: int, max_iter: int = 5000):
    """Lloyd-Max codebook of f_k on [0, π/2] with 2^bits levels (symmetric about
    π/4): boundaries are midpoints of neighbouring centroids, centroids are the
    conditional means of their cells.  Returns (centroids, bounds, mse)."""
    n = 1 << bits
    lo, hi = 0.0, np.pi / 2.0

    def mass(a, b):
        return float(angle_cdf(b, k) - angle_cdf(a, k))

    def moment(a, b):
        v, _ = integrate.quad(lambda p: p * angle_density(p, k), a, b, epsabs=1e-15, epsrel=1e-13, limit=200)
        return v

    # start from the conditional means of equal-probability cells
    qs = [lo] + [float(np.arcsin(np.sqrt(special.betaincinv(k / 2.0, k / 2.0, j / n)))) for j in range(1, n)] + [hi]
    c = np.array([moment(qs[j], qs[j + 1]) / mass(qs[j], qs[j + 1]) for j in range(n)])
    for _ in range(max_iter):
        t = [lo] + [0.5 * (c[j] + c[j + 1]) for j in range(n - 1)] + [hi]
        cn = np.array([moment(t[j], t[j + 1]) / max(mass(t[j], t[j + 1]), 1e-300) for j in range(n)])
        delta = float(np.max(np.abs(cn - c)))
        c = cn
        if delta <= 1e-13:
            break
    bounds = np.array([0.5 * (c[j] + c[j + 1]) for j in range(n - 1)])
    edges = np.concatenate([[lo], bounds, [hi]])
    mse = 0.0
    for j in range(n):
        v, _ = integrate.quad(lambda p: (p - c[j]) ** 2 * angle_density(p, k), edges[j], edges[j + 1],
                              epsabs=1e-15, epsrel=1e-12, limit=200)
        mse += v
    return c, bounds, mse


@dataclass
class PolarCodebooks:
    d: int
    b1: int
    b: int
    books: list  # per level: (centroids, bounds)


def make_codebooks(d: int, b1: int = 4, b: int = 2) -> PolarCodebooks:
    L = levels(d)
    books = [uniform_codebook(b1)]
    for lev in range(2, L + 1):
        c, bd, _ = lloyd_max_angle(1 << (lev - 1), b)
        books.append((c, bd))
    return PolarCodebooks(d=d, b1=b1, b=b, books=books)


@dataclass
class PolarQuantized:
    idx: list            # per level: [N, d/2^ℓ] int64 angle indices
    norm: np.ndarray     # [N] float32 ‖x‖
    sgn: np.ndarray      # [N, m] bool (QJL stage), True <-> +1
    rnorm: np.ndarray    # [N] float32 ‖r‖
    angles: list         # per level: exact angles (diagnostic)


def quantize_polar(X, Pi, S, cb: PolarCodebooks) -> PolarQuantized:
    """Rotate, polar-transform, quantize every angle with its level's codebook,
    then the QJL stage on the residual in the original domain."""
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=1))
    U = X @ Pi.T
    _, angles = forward(U)
    idx = [np.searchsorted(bd, ang, side="left").astype(np.int64) for (c, bd), ang in zip(cb.books, angles)]
    xt = reconstruct_stage1(idx, n, Pi, cb)
    r = X - xt
    p = r @ S.T if S.shape[0] > 0 else np.zeros((X.shape[0], 0))
    rn = np.sqrt(np.sum(r * r, axis=1))
    return PolarQuantized(idx=idx, norm=n.astype(np.float32), sgn=p >= 0.0, rnorm=rn.astype(np.float32),
                          angles=angles)


def reconstruct_stage1(idx, norm, Pi, cb: PolarCodebooks) -> np.ndarray:
    """x̃ = Πᵀ inverse(‖x‖, centroids of the stored angle indices)."""
    ang = [c[i] for (c, _), i in zip(cb.books, idx)]
    return inverse(np.asarray(norm, dtype=np.float64), ang) @ Pi


def reconstruct(q: PolarQuantized, Pi, S, cb: PolarCodebooks, qjl_stage: bool = True) -> np.ndarray:
    """x̂ = x̃ + √(π/2)/m ‖r‖ Sᵀσ from stored record values."""
    x = reconstruct_stage1(q.idx, q.norm, Pi, cb)
    if qjl_stage and S.shape[0] > 0:
        m = S.shape[0]
        sig = np.where(q.sgn, 1.0, -1.0)
        x = x + (math.sqrt(math.pi / 2.0) / m) * np.asarray(q.rnorm, dtype=np.float64)[:, None] * (sig @ S)
    return x


def bits_per_vector(d: int, b1: int = 4, b: int = 2) -> int:
    """Angle bits of one vector: d/2 level-1 angles at b1 bits, d/2 - 1 later ones at b."""
    return (d // 2) * b1 + (d // 2 - 1) * b


def index_words(d: int, b1: int = 4, b: int = 2) -> int:
    """32-bit words of one vector's angle codes (see pack_indices)."""
    return -(-(d // 2) * b1 // 32) + -(-(d // 2 - 1) * b // 32)


def pack_indices(idx, d: int, b1: int = 4, b: int = 2) -> np.ndarray:
    """Angle codes of N vectors -> [N, index_words] uint32.  The d/2 level-1
    codes (b1 bits) come first, 32/b1 to a word, code i at bits
    [b1·(i mod 32/b1), +b1) of word i // (32/b1) ("TurboQuant压缩效果": eight
    4-bit numbers in one 32-bit integer); then, from the next word on, the
    codes of levels 2, 3, ... in that order, b bits each, packed the same way."""
    N = idx[0].shape[0]
    out = np.zeros((N, index_words(d, b1, b)), dtype=np.uint64)
    first = np.asarray(idx[0], dtype=np.uint64)
    per1 = 32 // b1
    for i in range(d // 2):
        out[:, i // per1] |= first[:, i] << np.uint64(b1 * (i % per1))
    rest = np.concatenate([np.asarray(a, dtype=np.uint64) for a in idx[1:]], axis=1) if len(idx) > 1 else \
        np.zeros((N, 0), dtype=np.uint64)
    base = -(-(d // 2) * b1 // 32)
    per = 32 // b
    for i in range(rest.shape[1]):
        out[:, base + i // per] |= rest[:, i] << np.uint64(b * (i % per))
    return out.astype(np.uint32)


def unpack_indices(words, d: int, b1: int = 4, b: int = 2):
    """Inverse of pack_indices: list of per-level [N, d/2^ℓ] int64 codes."""
    w = np.asarray(words, dtype=np.uint64)
    per1, per = 32 // b1, 32 // b
    first = np.stack([(w[:, i // per1] >> np.uint64(b1 * (i % per1))) & np.uint64((1 << b1) - 1)
                      for i in range(d // 2)], axis=1).astype(np.int64)
    base = -(-(d // 2) * b1 // 32)
    rest = np.stack([(w[:, base + i // per] >> np.uint64(b * (i % per))) & np.uint64((1 << b) - 1)
                     for i in range(d // 2 - 1)], axis=1).astype(np.int64) if d > 2 else np.zeros((w.shape[0], 0),
                                                                                                 dtype=np.int64)
    out, off = [first], 0
    for lev in range(2, levels(d) + 1):
        n = d >> lev
        out.append(rest[:, off:off + n])
        off += n
    return out


def decode_attention_polar(q, K: PolarQuantized, V: PolarQuantized, shape, ctx_len, Pi, S, cb, scale=None):
    """Softmax attention over polar records; shape = (B, Hkv, T), rows in that order."""
    from .decode import attention

    B, Hkv, T = shape
    d = cb.d
    Kh = reconstruct(K, Pi, S, cb).reshape(B, Hkv, T, d)
    Vh = reconstruct(V, Pi, S, cb).reshape(B, Hkv, T, d)
    return attention(q, Kh, Vh, ctx_len, scale)
