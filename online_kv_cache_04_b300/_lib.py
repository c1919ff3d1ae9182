"""ctypes binding of libturboquant (argument marshalling only).

Every function here has the name of the C entry point it wraps and does no
arithmetic of its own: torch tensors supply device memory and streams, and
every step of the quantizer and the attention runs in the library's CUDA
kernels.  If the library is missing, ``load()`` raises: there is no fallback.
"""

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libturboquant.so")

TQ_OK, TQ_ERR_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_WORKSPACE, TQ_ERR_NUMERIC = 0, -1, -2, -3, -4, -5
TQ_F32, TQ_BF16 = 0, 1
TQ_LAYOUT_ROWS, TQ_LAYOUT_BLOCK32 = 0, 1

_c_double_p = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p


class tq_plan(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("m", ctypes.c_int), ("w", ctypes.c_int), ("qjl_alpha", ctypes.c_float),
                ("pi", _vp), ("pi_t", _vp), ("s_rot", _vp), ("s_rot_t", _vp), ("centroids", _vp),
                ("bounds", _vp), ("walsh", _vp), ("pi_bf16", _vp), ("s_bf16", _vp), ("pi_frag", _vp),
                ("s_frag", _vp), ("s_x_bf16", _vp)]


class tq_polar_plan(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("m", ctypes.c_int), ("b1", ctypes.c_int), ("b", ctypes.c_int),
                ("qjl_alpha", ctypes.c_float), ("pi", _vp), ("pi_t", _vp), ("s_rot", _vp), ("s_rot_t", _vp),
                ("tables", _vp)]


class tq_records(ctypes.Structure):
    _fields_ = [("idx", _vp), ("sgn", _vp), ("norm", _vp), ("rnorm", _vp), ("capacity", ctypes.c_int64),
                ("layout", ctypes.c_int32)]


# name -> (restype, argtypes)
_SIGNATURES = {
    "tq_make_rotation": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64, _c_double_p]),
    "tq_make_codebook": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _c_double_p, _c_double_p, _c_double_p]),
    "tq_make_qjl": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, _c_double_p, _c_double_p,
                                   _c_double_p]),
    "tq_plan_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_plan_init": (ctypes.c_int, [ctypes.POINTER(tq_plan), ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_double_p,
                                    _c_double_p, _c_double_p, _c_double_p, _vp, ctypes.c_size_t, _vp]),
    "tq_quantize": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.POINTER(tq_records), ctypes.c_int64, _vp]),
    "tq_quantize_pair": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, _vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.POINTER(tq_records), ctypes.POINTER(tq_records), ctypes.c_int64, _vp]),
    "tq_append_kv": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.POINTER(tq_records), ctypes.POINTER(tq_records), _vp, ctypes.c_int64,
                                    _vp]),
    "tq_decode_workspace_size": (ctypes.c_int, [ctypes.POINTER(tq_plan), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]),
    "tq_decode_attention": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(tq_records), ctypes.POINTER(tq_records), _vp,
                                           ctypes.c_int64, ctypes.c_float, _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_decode_attention_noalloc": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.POINTER(tq_records),
                                                   ctypes.POINTER(tq_records), _vp, ctypes.c_int64, ctypes.c_float,
                                                   _vp, _vp]),
    "tq_decode_scores": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.POINTER(tq_records), _vp, ctypes.c_int64, ctypes.c_float,
                                        _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_search_workspace_size": (ctypes.c_int, [ctypes.POINTER(tq_plan), ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_size_t)]),
    "tq_search_topk": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(tq_records), ctypes.c_int64, ctypes.c_int, _vp, _vp, _vp,
                                      ctypes.c_size_t, _vp]),
    "tq_quantize_split": (ctypes.c_int, [ctypes.POINTER(tq_plan), ctypes.POINTER(tq_plan), _vp, _vp, ctypes.c_int,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(tq_records),
                                         ctypes.POINTER(tq_records), ctypes.c_int64, _vp]),
    "tq_decode_split_workspace_size": (ctypes.c_int, [ctypes.POINTER(tq_plan), ctypes.POINTER(tq_plan), ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                      ctypes.POINTER(ctypes.c_size_t)]),
    "tq_decode_attention_split": (ctypes.c_int, [ctypes.POINTER(tq_plan), ctypes.POINTER(tq_plan), _vp, _vp, _vp,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(tq_records), ctypes.POINTER(tq_records),
                                                 ctypes.POINTER(tq_records), ctypes.POINTER(tq_records), _vp,
                                                 ctypes.c_int64, ctypes.c_float, _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_make_polar_codebooks": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _c_double_p, _c_double_p]),
    "tq_polar_index_words": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_polar_plan_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_polar_plan_init": (ctypes.c_int, [ctypes.POINTER(tq_polar_plan), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, _c_double_p, _c_double_p, _c_double_p, _c_double_p, _vp,
                                          ctypes.c_size_t, _vp]),
    "tq_quantize_polar": (ctypes.c_int, [ctypes.POINTER(tq_polar_plan), _vp, ctypes.c_int, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.POINTER(tq_records), ctypes.c_int64, _vp]),
    "tq_decode_polar_workspace_size": (ctypes.c_int, [ctypes.POINTER(tq_polar_plan), ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]),
    "tq_decode_attention_polar": (ctypes.c_int, [ctypes.POINTER(tq_polar_plan), _vp, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(tq_records),
                                                 ctypes.POINTER(tq_records), _vp, ctypes.c_int64, ctypes.c_float,
                                                 _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_decode_attention_paged": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(tq_records),
                                                 ctypes.POINTER(tq_records), _vp, _vp, ctypes.c_int, ctypes.c_float,
                                                 _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_append_kv_paged": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, _vp, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.POINTER(tq_records), ctypes.POINTER(tq_records), _vp,
                                          _vp, ctypes.c_int, _vp]),
    "tq_decode_attention_append": (ctypes.c_int, [ctypes.POINTER(tq_plan), _vp, ctypes.c_int, _vp, _vp, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(tq_records),
                                                  ctypes.POINTER(tq_records), _vp, ctypes.c_int64, _vp, ctypes.c_float,
                                                  _vp, _vp, ctypes.c_size_t, _vp]),
    "tq_fault_flags": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "tq_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def load():
    """Load libturboquant.so (built in-tree); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libturboquant.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class TQError(RuntimeError):
    def __init__(self, name, code):
        msg = load().tq_status_str(code).decode()
        super().__init__(f"{name} failed: {msg} ({code})")
        self.code = code


def _check(name, code):
    if code != TQ_OK:
        raise TQError(name, code)


def _dptr(a):
    return a.ctypes.data_as(_c_double_p) if a is not None else None


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _on_device(name, *tensors):
    """Device calls take CUDA tensors: a host pointer would reach a kernel and fault there."""
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name}: every tensor argument must live on a CUDA device")


def _records_on_device(name, *recs):
    for r in recs:
        _on_device(name, r.idx, r.sgn, r.norm, r.rnorm)


def _lengths(name, ctx_len):
    import torch

    _on_device(name, ctx_len)
    if ctx_len.dtype != torch.int32:
        raise ValueError(f"{name}: ctx_len must be int32")


def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return TQ_F32
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------- host setup

def tq_make_rotation(d, seed):
    pi = np.empty((d, d), dtype=np.float64)
    _check("tq_make_rotation", load().tq_make_rotation(d, seed, _dptr(pi)))
    return pi


def tq_make_codebook(d, w):
    c = np.empty(1 << w, dtype=np.float64)
    b = np.empty((1 << w) - 1, dtype=np.float64)
    mse = np.empty(1, dtype=np.float64)
    _check("tq_make_codebook", load().tq_make_codebook(d, w, _dptr(c), _dptr(b), _dptr(mse)))
    return c, b, float(mse[0])


def tq_make_qjl(m, d, seed, pi=None):
    S = np.empty((m, d), dtype=np.float64)
    s_rot = np.empty((m, d), dtype=np.float64) if pi is not None else None
    pi_c = np.ascontiguousarray(pi, dtype=np.float64) if pi is not None else None
    _check("tq_make_qjl", load().tq_make_qjl(m, d, seed, _dptr(pi_c), _dptr(S), _dptr(s_rot)))
    return S, s_rot


# ----------------------------------------------------------------- device objects

class Plan:
    """Device tables of one (d, m, w) shape: a tq_plan over a torch buffer."""

    def __init__(self, d, m, w, rotation_seed, qjl_seed, device="cuda", stream=None):
        import torch

        self.d, self.m, self.w = d, m, w
        self.pi = tq_make_rotation(d, rotation_seed)
        # m = 0: stage 1 alone, no QJL matrix
        self.S, self.s_rot = tq_make_qjl(m, d, qjl_seed, self.pi) if m > 0 else (np.zeros((0, d)), None)
        self.centroids, self.bounds, self.mse = tq_make_codebook(d, w)
        nbytes = load().tq_plan_bytes(d, m, w)
        if nbytes == 0:
            raise TQError("tq_plan_bytes", TQ_ERR_ARG)
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.c = tq_plan()
        _check("tq_plan_init", load().tq_plan_init(
            ctypes.byref(self.c), d, m, w, _dptr(self.pi), _dptr(self.s_rot), _dptr(self.centroids),
            _dptr(self.bounds), self.buffer.data_ptr(), nbytes, _stream(stream)))

    @property
    def ref(self):
        return ctypes.byref(self.c)


class Records:
    """Compressed vectors (SoA) in torch device tensors.

    layout TQ_LAYOUT_ROWS: one row of bit words per vector; TQ_LAYOUT_BLOCK32:
    32-row blocks with one coordinate per word (the value-cache layout of the
    tensor-core decode; capacity a multiple of 32).  Both hold the same bytes.
    """

    def __init__(self, capacity, d, m, w, device="cuda", layout=TQ_LAYOUT_ROWS):
        import torch

        self.capacity, self.d, self.m, self.w, self.layout = capacity, d, m, w, layout
        self.idx = torch.empty(capacity, w * d // 32, dtype=torch.int32, device=device)
        self.norm = torch.empty(capacity, dtype=torch.float32, device=device)
        # stage-1-only records (m = 0) carry no signs and no residual norm
        self.sgn = torch.empty(capacity, m // 32, dtype=torch.int32, device=device) if m > 0 else None
        self.rnorm = torch.empty(capacity, dtype=torch.float32, device=device) if m > 0 else None
        self.c = tq_records(self.idx.data_ptr(), self.sgn.data_ptr() if m > 0 else None, self.norm.data_ptr(),
                            self.rnorm.data_ptr() if m > 0 else None, capacity, layout)

    @classmethod
    def wrap(cls, idx, sgn, norm, rnorm, d, m, w, layout=TQ_LAYOUT_ROWS):
        """Records over existing tensors (e.g. the oracle's packed words)."""
        self = cls.__new__(cls)
        self.capacity, self.d, self.m, self.w, self.layout = norm.shape[0], d, m, w, layout
        self.idx, self.sgn, self.norm, self.rnorm = idx, sgn, norm, rnorm
        ptr = lambda t: None if t is None else t.data_ptr()
        self.c = tq_records(idx.data_ptr(), ptr(sgn), norm.data_ptr(), ptr(rnorm), self.capacity, layout)
        return self

    @property
    def ref(self):
        return ctypes.byref(self.c)


# ----------------------------------------------------------------- device calls

def tq_quantize(plan, x, out, out_offset=0, stream=None):
    """Quantize the rows of x [n, ld>=d] (fp32 or bf16, device) into out[out_offset:]."""
    _on_device("tq_quantize", x)
    _records_on_device("tq_quantize", out)
    n = x.shape[0]
    ld = x.stride(0) if x.dim() == 2 and n > 0 else plan.d
    _check("tq_quantize", load().tq_quantize(plan.ref, x.data_ptr(), _dtype_code(x), n, ld, out.ref, out_offset,
                                             _stream(stream)))


def tq_quantize_pair(plan, x0, x1, out0, out1, out_offset=0, stream=None):
    """Quantize x0 into out0 and x1 into out1 (same shape, dtype and row stride), rows out_offset onward."""
    _on_device("tq_quantize_pair", x0, x1)
    _records_on_device("tq_quantize_pair", out0, out1)
    if x0.shape != x1.shape or x0.dtype != x1.dtype or x0.stride() != x1.stride():
        raise ValueError("tq_quantize_pair: x0 and x1 must have the same shape, dtype and strides")
    n = x0.shape[0]
    ld = x0.stride(0) if x0.dim() == 2 and n > 0 else plan.d
    _check("tq_quantize_pair", load().tq_quantize_pair(plan.ref, x0.data_ptr(), x1.data_ptr(), _dtype_code(x0), n, ld,
                                                       out0.ref, out1.ref, out_offset, _stream(stream)))


def tq_append_kv(plan, k_new, v_new, K, V, ctx_len, ctx_stride, stream=None):
    """Store the new key and value of every (batch row, kv head) at token ctx_len[b] and advance ctx_len.

    k_new, v_new: device [B, Hkv, d] (fp32 or bf16, contiguous); ctx_len: device int32 [B], updated in place.
    """
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype or k_new.dim() != 3:
        raise ValueError("tq_append_kv: k_new and v_new must both be [B, Hkv, d] of one dtype")
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("tq_append_kv: k_new and v_new must be contiguous")
    import torch

    if ctx_len.dtype != torch.int32 or ctx_len.numel() != k_new.shape[0]:
        raise ValueError("tq_append_kv: ctx_len must be int32 [B]")
    _on_device("tq_append_kv", k_new, v_new, ctx_len)
    _records_on_device("tq_append_kv", K, V)
    B, Hkv, _ = k_new.shape
    _check("tq_append_kv", load().tq_append_kv(plan.ref, k_new.data_ptr(), v_new.data_ptr(), _dtype_code(k_new), B,
                                               Hkv, K.ref, V.ref, ctx_len.data_ptr(), ctx_stride, _stream(stream)))


def tq_decode_workspace_size(plan, B, Hq, Hkv, ctx_stride):
    n = ctypes.c_size_t(0)
    _check("tq_decode_workspace_size", load().tq_decode_workspace_size(plan.ref, B, Hq, Hkv, ctx_stride,
                                                                       ctypes.byref(n)))
    return n.value


def tq_decode_attention(plan, q, K, V, ctx_len, ctx_stride, Hkv, out, workspace, scale=0.0, stream=None):
    _on_device("tq_decode_attention", q, out, workspace)
    _lengths("tq_decode_attention", ctx_len)
    _records_on_device("tq_decode_attention", K, V)
    B, Hq, _ = q.shape
    _check("tq_decode_attention", load().tq_decode_attention(
        plan.ref, q.data_ptr(), _dtype_code(q), B, Hq, Hkv, K.ref, V.ref, ctx_len.data_ptr(), ctx_stride,
        float(scale), out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def tq_decode_attention_noalloc(plan, q, K, V, ctx_len, ctx_stride, Hkv, out, scale=0.0, stream=None):
    """tq_decode_attention with the library's built-in scratch array (no workspace argument)."""
    _on_device("tq_decode_attention_noalloc", q, out)
    _lengths("tq_decode_attention_noalloc", ctx_len)
    _records_on_device("tq_decode_attention_noalloc", K, V)
    B, Hq, _ = q.shape
    _check("tq_decode_attention_noalloc", load().tq_decode_attention_noalloc(
        plan.ref, q.data_ptr(), _dtype_code(q), B, Hq, Hkv, K.ref, V.ref, ctx_len.data_ptr(), ctx_stride,
        float(scale), out.data_ptr(), _stream(stream)))


def tq_decode_attention_paged(plan, q, K, V, ctx_len, pages, Hkv, out, workspace, scale=0.0, stream=None):
    """Decode over paged caches: pages [B*Hkv, max_pages] int32 (device), 256 tokens per page."""
    _on_device("tq_decode_attention_paged", q, out, workspace, pages)
    _lengths("tq_decode_attention_paged", ctx_len)
    _records_on_device("tq_decode_attention_paged", K, V)
    B, Hq, _ = q.shape
    _check("tq_decode_attention_paged", load().tq_decode_attention_paged(
        plan.ref, q.data_ptr(), _dtype_code(q), B, Hq, Hkv, K.ref, V.ref, ctx_len.data_ptr(), pages.data_ptr(),
        pages.shape[-1], float(scale), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_decode_attention_append(plan, q, k_new, v_new, K, V, ctx_len, ctx_stride, Hkv, out, workspace, pages=None,
                               scale=0.0, stream=None):
    """One decode step with the append fused in: store k_new, v_new ([B, Hkv, d]) at token ctx_len[b], attend over
    ctx_len[b] + 1 tokens, advance ctx_len.  pages: None (contiguous caches) or [B*Hkv, ctx_stride / 256] int32."""
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype or k_new.dim() != 3:
        raise ValueError("tq_decode_attention_append: k_new and v_new must both be [B, Hkv, d] of one dtype")
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("tq_decode_attention_append: k_new and v_new must be contiguous")
    _on_device("tq_decode_attention_append", q, k_new, v_new, out, workspace)
    _lengths("tq_decode_attention_append", ctx_len)
    _records_on_device("tq_decode_attention_append", K, V)
    if pages is not None:
        _on_device("tq_decode_attention_append", pages)
    B, Hq, _ = q.shape
    _check("tq_decode_attention_append", load().tq_decode_attention_append(
        plan.ref, q.data_ptr(), _dtype_code(q), k_new.data_ptr(), v_new.data_ptr(), _dtype_code(k_new), B, Hq, Hkv,
        K.ref, V.ref, ctx_len.data_ptr(), ctx_stride, None if pages is None else pages.data_ptr(), float(scale),
        out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_append_kv_paged(plan, k_new, v_new, K, V, ctx_len, pages, stream=None):
    """tq_append_kv into paged caches (pages [B*Hkv, max_pages] int32, device)."""
    if k_new.shape != v_new.shape or k_new.dtype != v_new.dtype or k_new.dim() != 3:
        raise ValueError("tq_append_kv_paged: k_new and v_new must both be [B, Hkv, d] of one dtype")
    if not (k_new.is_contiguous() and v_new.is_contiguous() and pages.is_contiguous()):
        raise ValueError("tq_append_kv_paged: k_new, v_new and pages must be contiguous")
    _on_device("tq_append_kv_paged", k_new, v_new, pages)
    _lengths("tq_append_kv_paged", ctx_len)
    _records_on_device("tq_append_kv_paged", K, V)
    B, Hkv, _ = k_new.shape
    _check("tq_append_kv_paged", load().tq_append_kv_paged(
        plan.ref, k_new.data_ptr(), v_new.data_ptr(), _dtype_code(k_new), B, Hkv, K.ref, V.ref, ctx_len.data_ptr(),
        pages.data_ptr(), pages.shape[-1], _stream(stream)))


def tq_decode_scores(plan, q, K, ctx_len, ctx_stride, Hkv, scores, workspace, scale=0.0, stream=None):
    _on_device("tq_decode_scores", q, scores, workspace)
    _lengths("tq_decode_scores", ctx_len)
    _records_on_device("tq_decode_scores", K)
    B, Hq, _ = q.shape
    _check("tq_decode_scores", load().tq_decode_scores(
        plan.ref, q.data_ptr(), _dtype_code(q), B, Hq, Hkv, K.ref, ctx_len.data_ptr(), ctx_stride, float(scale),
        scores.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_search_workspace_size(plan, nq, n, k):
    b = ctypes.c_size_t(0)
    _check("tq_search_workspace_size", load().tq_search_workspace_size(plan.ref, nq, n, k, ctypes.byref(b)))
    return b.value


def tq_search_topk(plan, q, recs, n, k, idx_out, score_out, workspace, stream=None):
    _on_device("tq_search_topk", q, idx_out, score_out, workspace)
    _records_on_device("tq_search_topk", recs)
    _check("tq_search_topk", load().tq_search_topk(
        plan.ref, q.data_ptr(), _dtype_code(q), q.shape[0], recs.ref, n, k, idx_out.data_ptr(),
        score_out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_quantize_split(plan_o, plan_r, perm, x, out_o, out_r, out_offset=0, stream=None):
    """Outlier channels perm[:plan_o.d] of each row of x [n, ld>=d] through plan_o into out_o,
    the rest through plan_r into out_r.  perm: device int32 [d]."""
    _on_device("tq_quantize_split", x, perm)
    _records_on_device("tq_quantize_split", out_o, out_r)
    import torch

    if perm.dtype != torch.int32:
        raise ValueError("tq_quantize_split: perm must be int32")
    n = x.shape[0]
    ld = x.stride(0) if x.dim() == 2 and n > 0 else plan_o.d + plan_r.d
    _check("tq_quantize_split", load().tq_quantize_split(plan_o.ref, plan_r.ref, perm.data_ptr(), x.data_ptr(),
                                                         _dtype_code(x), n, ld, out_o.ref, out_r.ref, out_offset,
                                                         _stream(stream)))


def tq_decode_split_workspace_size(plan_o, plan_r, B, Hq, Hkv, ctx_stride):
    n = ctypes.c_size_t(0)
    _check("tq_decode_split_workspace_size", load().tq_decode_split_workspace_size(
        plan_o.ref, plan_r.ref, B, Hq, Hkv, ctx_stride, ctypes.byref(n)))
    return n.value


def tq_decode_attention_split(plan_o, plan_r, perm_k, perm_v, q, K_o, K_r, V_o, V_r, ctx_len, ctx_stride, Hkv, out,
                              workspace, scale=0.0, stream=None):
    _on_device("tq_decode_attention_split", perm_k, perm_v, q, out, workspace)
    _lengths("tq_decode_attention_split", ctx_len)
    _records_on_device("tq_decode_attention_split", K_o, K_r, V_o, V_r)
    B, Hq, _ = q.shape
    _check("tq_decode_attention_split", load().tq_decode_attention_split(
        plan_o.ref, plan_r.ref, perm_k.data_ptr(), perm_v.data_ptr(), q.data_ptr(), _dtype_code(q), B, Hq, Hkv,
        K_o.ref, K_r.ref, V_o.ref,
        V_r.ref, ctx_len.data_ptr(), ctx_stride, float(scale), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_make_polar_codebooks(d, b1=4, b=2):
    """Per-level (centroids, bounds) lists, float64."""
    L = int(d).bit_length() - 1
    c = np.empty((1 << b1) + (L - 1) * (1 << b), dtype=np.float64)
    bd = np.empty(((1 << b1) - 1) + (L - 1) * ((1 << b) - 1), dtype=np.float64)
    _check("tq_make_polar_codebooks", load().tq_make_polar_codebooks(d, b1, b, _dptr(c), _dptr(bd)))
    books = [(c[:1 << b1], bd[:(1 << b1) - 1])]
    for lev in range(L - 1):
        o, ob = (1 << b1) + lev * (1 << b), ((1 << b1) - 1) + lev * ((1 << b) - 1)
        books.append((c[o:o + (1 << b)], bd[ob:ob + (1 << b) - 1]))
    return books, c, bd


class PolarPlan:
    """Device tables of the polar stage of one (d, m, b1, b) shape."""

    def __init__(self, d, m, b1, b, rotation_seed, qjl_seed, device="cuda", stream=None):
        import torch

        self.d, self.m, self.b1, self.b = d, m, b1, b
        self.pi = tq_make_rotation(d, rotation_seed)
        self.S, self.s_rot = tq_make_qjl(m, d, qjl_seed, self.pi)
        self.books, c, bd = tq_make_polar_codebooks(d, b1, b)
        self.nw = load().tq_polar_index_words(d, b1, b)
        nbytes = load().tq_polar_plan_bytes(d, m, b1, b)
        if nbytes == 0 or self.nw == 0:
            raise TQError("tq_polar_plan_bytes", TQ_ERR_ARG)
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.c = tq_polar_plan()
        _check("tq_polar_plan_init", load().tq_polar_plan_init(
            ctypes.byref(self.c), d, m, b1, b, _dptr(self.pi), _dptr(self.s_rot), _dptr(c), _dptr(bd),
            self.buffer.data_ptr(), nbytes, _stream(stream)))

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def records(self, capacity, device="cuda"):
        """Polar records of `capacity` rows (TQ_LAYOUT_ROWS)."""
        import torch

        idx = torch.empty(capacity, self.nw, dtype=torch.int32, device=device)
        sgn = torch.empty(capacity, self.m // 32, dtype=torch.int32, device=device)
        norm = torch.empty(capacity, dtype=torch.float32, device=device)
        rnorm = torch.empty(capacity, dtype=torch.float32, device=device)
        return Records.wrap(idx, sgn, norm, rnorm, self.d, self.m, 0)


def tq_quantize_polar(plan, x, out, out_offset=0, stream=None):
    _on_device("tq_quantize_polar", x)
    _records_on_device("tq_quantize_polar", out)
    n = x.shape[0]
    ld = x.stride(0) if x.dim() == 2 and n > 0 else plan.d
    _check("tq_quantize_polar", load().tq_quantize_polar(plan.ref, x.data_ptr(), _dtype_code(x), n, ld, out.ref,
                                                         out_offset, _stream(stream)))


def tq_decode_polar_workspace_size(plan, B, Hq, Hkv, ctx_stride):
    n = ctypes.c_size_t(0)
    _check("tq_decode_polar_workspace_size", load().tq_decode_polar_workspace_size(plan.ref, B, Hq, Hkv, ctx_stride,
                                                                                   ctypes.byref(n)))
    return n.value


def tq_decode_attention_polar(plan, q, K, V, ctx_len, ctx_stride, Hkv, out, workspace, scale=0.0, stream=None):
    _on_device("tq_decode_attention_polar", q, out, workspace)
    _lengths("tq_decode_attention_polar", ctx_len)
    _records_on_device("tq_decode_attention_polar", K, V)
    B, Hq, _ = q.shape
    _check("tq_decode_attention_polar", load().tq_decode_attention_polar(
        plan.ref, q.data_ptr(), _dtype_code(q), B, Hq, Hkv, K.ref, V.ref, ctx_len.data_ptr(), ctx_stride,
        float(scale), out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def tq_fault_flags(reset=True):
    """Device fault bits: bounded waits that ran out, appends to a full cache (0 = none)."""
    v = ctypes.c_uint32(0)
    _check("tq_fault_flags", load().tq_fault_flags(ctypes.byref(v), 1 if reset else 0))
    return v.value
