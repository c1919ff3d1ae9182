"""Plain float64 CPU oracle for the TurboQuant hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The library (``online_kv_cache_04_b300``) never imports it, and this
package imports nothing from the library: the two share no code, tables or
constants.  Inputs reach both sides from the seeded generators in
``online_kv_cache_04_b300.workloads``, which hold none of the method's
arithmetic.

Every function follows the published description step by step, in NumPy /
SciPy float64, with no blocking, fusion or reordering.  Sources are cited by
page title and section:

* [memory-wall] "谷歌TurboQuant如何绕过内存墙？重新审视它的技术突破"
  (youleyou), §2 "TurboQuant到底做了什么？": stage 1 (random rotation + Lloyd-Max
  scalar quantizer for the Beta coordinate law), stage 2 (1-bit QJL on the
  residual), the 2/π bias remark and the MSE bounds.
* [efficiency] "TurboQuant 与 AI 效率革命：当旧数学遇到新智能" (mini-blog),
  §三 "补刀：1-bit 的极限操作" (JL transform, asymmetric estimator, bit
  accounting) and §四 "整合：TurboQuant 的三段论" (three-step pipeline).
* [video] "TurboQuant压缩效果" (douyin transcripts): fused operators that read
  packed words and decode in registers; several small codes per 32-bit word.
* [yeyu] yeyulingfeng article: codebook computed once, no calibration.

Modules
-------
prng       SplitMix64 counter generator + Box-Muller normals
rotation   Haar rotation Π from Gaussian QR (u = Π x)
codebook   Lloyd-Max codebook for f_d(x) ∝ (1-x²)^((d-3)/2)
qjl        Gaussian JL matrix S and the asymmetric sign estimator
quantize   the two-stage quantizer (rotate, bucketize, residual, QJL signs)
pack       bit-sliced packing of indices and signs into 32-bit words
decode     scores and softmax attention over stored records
search     inner-product top-k over stored records
mixed      outlier-channel split precision (two instances, b + 1 / b bits)
polar      PolarQuant's recursive polar stage, an alternative stage 1
"""

from . import prng, rotation, codebook, qjl, quantize, pack, decode, search, mixed, polar  # noqa: F401
