"""TurboQuant online KV-vector quantization and compressed-cache decode attention
for NVIDIA B300 (sm_103a).

The compute lives in ``libturboquant.so`` (CUDA kernels behind a C ABI,
declared in ``include/turboquant.h``).  ``_lib`` is a thin ctypes binding with
the same names; ``workloads`` draws the seeded synthetic inputs.
"""

from ._lib import (Plan, PolarPlan, Records, TQError, load, tq_append_kv, tq_append_kv_paged,  # noqa: F401
                   tq_decode_attention, tq_decode_attention_append, tq_decode_attention_noalloc,
                   tq_decode_attention_paged, tq_decode_attention_polar, tq_decode_attention_split, tq_decode_scores,
                   tq_decode_workspace_size, tq_fault_flags, tq_make_codebook, tq_make_qjl, tq_make_rotation,
                   tq_quantize, tq_quantize_pair, tq_quantize_polar, tq_quantize_split, tq_search_topk,
                   tq_search_workspace_size)
