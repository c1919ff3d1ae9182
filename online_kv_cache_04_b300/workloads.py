"""Seeded synthetic workloads (shapes and value laws of the published workloads).

This module only draws inputs: it holds none of the quantizer's or the
attention's arithmetic, so both the CUDA path and the float64 oracle can be
fed from it.  The pages measure on LongBench / needle-in-a-haystack with
Llama-3.1-8B-class models; no dataset or weights are used here, only tensors
of the same shapes with heavy-tailed per-channel scales and outlier channels,
the case that motivates the random rotation.

Workloads (all d = head_dim, m = QJL rows = d):

* ``tiny``      one kv head, d=128, 4096 keys+values fp32 ~N(0,1) with 4
                outlier channels x10, b=3, 8 fp32 queries (8 query heads).
* ``llama8b``   Llama-3.1-8B decode layer: 32 query / 8 kv heads, d=128,
                batch 1, context 32768, bf16 K/V = N(0,1)·s_c with
                s_c ~ LogNormal(0, 1) per (kv head, channel), independent for
                K and V, 4 outlier channels x20; b in {3, 4}.
* ``longctx``   batch 16, context 131072, same law, b in {2, 3, 4}.
* ``prefill``   8 kv heads x 65536 tokens x {K, V} bf16 (1,048,576 vectors),
                same law, b=3.
* ``generic``   1,048,576 unit-norm fp32 vectors, d=1024, Gaussian with
                eigenvalues ∝ 1/i, b=4, m=1024; 1024 queries of the same law.
"""

from dataclasses import dataclass, field

import torch

ROTATION_SEED = 0x71550001
QJL_SEED = 0x71550002
# split precision: the outlier side's and the regular side's own instances
SPLIT_SEEDS = {"outlier": (0x71550011, 0x71550012), "regular": (0x71550021, 0x71550022)}
# the polar stage's rotation and QJL matrix
POLAR_SEEDS = (0x71550031, 0x71550032)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    m: int
    ctx: int
    bits: tuple
    dtype: torch.dtype
    outlier_scale: float
    lognormal_sigma: float
    data_seed: int
    n_queries: int = 0  # search workloads only
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=8, Hkv=1, d=128, m=128, ctx=4096, bits=(3,), dtype=torch.float32,
                     outlier_scale=10.0, lognormal_sigma=0.0, data_seed=1001),
    "llama8b": Workload("llama8b", B=1, Hq=32, Hkv=8, d=128, m=128, ctx=32768, bits=(3, 4),
                        dtype=torch.bfloat16, outlier_scale=20.0, lognormal_sigma=1.0, data_seed=1002),
    "longctx": Workload("longctx", B=16, Hq=32, Hkv=8, d=128, m=128, ctx=131072, bits=(2, 3, 4),
                        dtype=torch.bfloat16, outlier_scale=20.0, lognormal_sigma=1.0, data_seed=1003),
    "prefill": Workload("prefill", B=1, Hq=32, Hkv=8, d=128, m=128, ctx=65536, bits=(3,),
                        dtype=torch.bfloat16, outlier_scale=20.0, lognormal_sigma=1.0, data_seed=1004),
    "generic": Workload("generic", B=1, Hq=1, Hkv=1, d=1024, m=1024, ctx=1048576, bits=(4,),
                        dtype=torch.float32, outlier_scale=1.0, lognormal_sigma=0.0, data_seed=1005,
                        n_queries=1024),
}


def channel_scales(Hkv: int, d: int, seed: int, lognormal_sigma: float, outlier_scale: float,
                   n_outliers: int = 4) -> torch.Tensor:
    """[Hkv, d] float32 per-channel scales: LogNormal(0, σ) times outlier factors."""
    g = torch.Generator().manual_seed(seed)
    if lognormal_sigma > 0.0:
        s = torch.exp(lognormal_sigma * torch.randn(Hkv, d, generator=g, dtype=torch.float64))
    else:
        s = torch.ones(Hkv, d, dtype=torch.float64)
    for h in range(Hkv):
        ch = torch.randperm(d, generator=g)[:n_outliers]
        s[h, ch] *= outlier_scale
    return s.float()


def make_kv(wl: Workload, B: int = None, T: int = None, which: int = 0, device="cpu",
            dtype: torch.dtype = None) -> torch.Tensor:
    """K (which=0) or V (which=1) cache [B, Hkv, T, d] of the workload's law.

    Rows are N(0, 1) · scale[h, c].  Generated on ``device`` with a generator
    seeded from the workload, so CPU and GPU draws differ: feed the oracle
    from the same tensor the GPU sees.
    """
    B = wl.B if B is None else B
    T = wl.ctx if T is None else T
    dtype = wl.dtype if dtype is None else dtype
    base = wl.data_seed * 16 + 2 * which
    scales = channel_scales(wl.Hkv, wl.d, base, wl.lognormal_sigma, wl.outlier_scale).to(device)
    g = torch.Generator(device=device).manual_seed(base + 1)
    x = torch.randn(B, wl.Hkv, T, wl.d, generator=g, device=device, dtype=torch.float32)
    x.mul_(scales[None, :, None, :])
    return x.to(dtype)


def make_queries(wl: Workload, B: int = None, device="cpu", dtype: torch.dtype = None) -> torch.Tensor:
    """q [B, Hq, d] ~ N(0, 1)."""
    B = wl.B if B is None else B
    dtype = wl.dtype if dtype is None else dtype
    g = torch.Generator(device=device).manual_seed(wl.data_seed * 16 + 5)
    return torch.randn(B, wl.Hq, wl.d, generator=g, device=device, dtype=torch.float32).to(dtype)


def make_anisotropic_unit(n: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """n unit-norm fp32 rows of z ~ N(0, diag(λ)), λ_i ∝ 1/i (standard basis)."""
    g = torch.Generator(device=device).manual_seed(seed)
    lam_sqrt = torch.rsqrt(torch.arange(1, d + 1, device=device, dtype=torch.float32))
    z = torch.randn(n, d, generator=g, device=device, dtype=torch.float32) * lam_sqrt
    return z / torch.linalg.vector_norm(z, dim=1, keepdim=True)


def make_generic(wl: Workload, n: int = None, device="cpu") -> torch.Tensor:
    return make_anisotropic_unit(wl.ctx if n is None else n, wl.d, wl.data_seed * 16, device)


def make_generic_queries(wl: Workload, nq: int = None, device="cpu") -> torch.Tensor:
    return make_anisotropic_unit(wl.n_queries if nq is None else nq, wl.d, wl.data_seed * 16 + 7, device)
