"""Python binding of ``libkda.so`` (argument marshalling only).

The raw functions below carry the C names and argument lists of ``include/kda.h`` and
take device pointers as integers. :func:`chunk_kda_fwd` is the convenience call on torch
CUDA tensors: it checks shapes and dtypes, allocates the outputs with torch and calls
the C ABI on the current torch stream. Every step of the computation runs in the
library's CUDA kernels; there is no other code path. If the library cannot be loaded
the import fails.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_ALIGNMENT = -3
KDA_ERR_CUDA = -4
KDA_DTYPE_BF16 = 0
KDA_DTYPE_F32 = 1
KDA_GATE_PER_CHANNEL = 0
KDA_GATE_PER_HEAD = 1
KDA_FLAG_ONE_CTA_PER_UNIT = 1
KDA_FLAG_UNFUSED_FRONTEND = 2
KDA_FLAG_DEBUG_SHORT_WAITS = 4
KDA_DEVICE_ERR_SEQLENS = 1
KDA_DEVICE_ERR_TIMEOUT = 2

EXPORTED = ("kda_chunk_fwd", "kda_chunk_fwd_f32", "kda_chunk_fwd_ex", "kda_status_string",
            "kda_get_device_error", "kda_chunk_fwd_noalloc", "kda_recurrent_fwd",
            "kda_recurrent_fwd_ex", "kda_chunk_fwd_fused", "kda_recurrent_fwd_fused",
            "kda_chunk_bwd")


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


class kda_fwd_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("ht", ctypes.c_void_p),
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H_k", ctypes.c_int), ("H_v", ctypes.c_int),
        ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("C", ctypes.c_int),
        ("scale", ctypes.c_float), ("cu_seqlens", ctypes.c_void_p),
        ("dtype", ctypes.c_int), ("gate_mode", ctypes.c_int), ("flags", ctypes.c_int),
    ]


class kda_bwd_params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("dO", ctypes.c_void_p), ("dht", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("dg", ctypes.c_void_p), ("dbeta", ctypes.c_void_p), ("dh0", ctypes.c_void_p),
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H_k", ctypes.c_int), ("H_v", ctypes.c_int),
        ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("C", ctypes.c_int),
        ("scale", ctypes.c_float), ("cu_seqlens", ctypes.c_void_p),
        ("dtype", ctypes.c_int), ("gate_mode", ctypes.c_int), ("flags", ctypes.c_int),
    ]


class kda_frontend(ctypes.Structure):
    _fields_ = [
        ("qk_l2norm", ctypes.c_int), ("beta_sigmoid", ctypes.c_int),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load ``libkda.so`` (building it first if it is missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build()
        if not os.path.exists(path):
            raise ImportError(f"libkda.so is missing at {path}")
        L = ctypes.CDLL(path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        sig = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P]
        for name in ("kda_chunk_fwd", "kda_chunk_fwd_f32", "kda_chunk_fwd_noalloc"):
            fn = getattr(L, name)
            fn.argtypes = sig
            fn.restype = I
        L.kda_chunk_fwd_ex.argtypes = [ctypes.POINTER(kda_fwd_params), P]
        L.kda_chunk_fwd_ex.restype = I
        L.kda_recurrent_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P]
        L.kda_recurrent_fwd.restype = I
        L.kda_recurrent_fwd_ex.argtypes = [ctypes.POINTER(kda_fwd_params), P]
        L.kda_recurrent_fwd_ex.restype = I
        L.kda_chunk_bwd.argtypes = [ctypes.POINTER(kda_bwd_params), P]
        L.kda_chunk_bwd.restype = I
        for name in ("kda_chunk_fwd_fused", "kda_recurrent_fwd_fused"):
            fn = getattr(L, name)
            fn.argtypes = [ctypes.POINTER(kda_fwd_params), ctypes.POINTER(kda_frontend), P]
            fn.restype = I
        L.kda_status_string.argtypes = [I]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_get_device_error.argtypes = [P]
        L.kda_get_device_error.restype = I
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


# ---- raw C entry points (pointers as ints, 0 for NULL) -----------------------------------

def kda_chunk_fwd(q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, C, scale, cu_seqlens,
                  stream) -> int:
    return lib().kda_chunk_fwd(q, k, v, g, beta, h0 or None, o, ht or None, B, T, H_k, H_v, d_k,
                               d_v, C, scale, cu_seqlens or None, stream or None)


def kda_chunk_fwd_f32(q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, C, scale, cu_seqlens,
                      stream) -> int:
    return lib().kda_chunk_fwd_f32(q, k, v, g, beta, h0 or None, o, ht or None, B, T, H_k, H_v,
                                   d_k, d_v, C, scale, cu_seqlens or None, stream or None)


def kda_chunk_fwd_noalloc(q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, C, scale,
                          cu_seqlens, stream) -> int:
    return lib().kda_chunk_fwd_noalloc(q, k, v, g, beta, h0 or None, o, ht or None, B, T, H_k, H_v,
                                       d_k, d_v, C, scale, cu_seqlens or None, stream or None)


def kda_chunk_fwd_ex(params: kda_fwd_params, stream) -> int:
    return lib().kda_chunk_fwd_ex(ctypes.byref(params), stream or None)


def kda_recurrent_fwd(q, k, v, g, beta, h0, o, ht, B, T, H_k, H_v, d_k, d_v, scale, cu_seqlens,
                      stream) -> int:
    return lib().kda_recurrent_fwd(q, k, v, g, beta or None, h0 or None, o, ht or None, B, T, H_k,
                                   H_v, d_k, d_v, scale, cu_seqlens or None, stream or None)


def kda_recurrent_fwd_ex(params: kda_fwd_params, stream) -> int:
    return lib().kda_recurrent_fwd_ex(ctypes.byref(params), stream or None)


def kda_chunk_fwd_fused(params: kda_fwd_params, fe: kda_frontend | None, stream) -> int:
    return lib().kda_chunk_fwd_fused(ctypes.byref(params), None if fe is None else ctypes.byref(fe),
                                     stream or None)


def kda_recurrent_fwd_fused(params: kda_fwd_params, fe: kda_frontend | None, stream) -> int:
    return lib().kda_recurrent_fwd_fused(ctypes.byref(params), None if fe is None else ctypes.byref(fe),
                                         stream or None)


def kda_chunk_bwd(params: kda_bwd_params, stream) -> int:
    return lib().kda_chunk_bwd(ctypes.byref(params), stream or None)


def kda_get_device_error(stream) -> int:
    return lib().kda_get_device_error(stream or None)


# ---- torch convenience ---------------------------------------------------------------------

def _ptr(t):
    return 0 if t is None else t.data_ptr()


def chunk_kda_fwd(q, k, v, g, beta, *, h0=None, scale=None, cu_seqlens=None,
                  output_final_state=True, chunk_size=64, o=None, ht=None, stream=None,
                  one_cta_per_unit=False, recurrent=False, qk_l2norm=False, beta_sigmoid=False,
                  A_log=None, dt_bias=None, unfused_frontend=False):
    """Chunkwise KDA forward on torch CUDA tensors; returns ``(o, ht)``.

    q, k [B, T, H_k, d_k] and v [B, T, H_v, d_v], all bf16 or all fp32; g fp32
    [B, T, H_v, d_k] (per-channel gate) or [B, T, H_v] (one gate per head); beta fp32
    [B, T, H_v], or None for the decay-only recurrence S <- Diag(a_t) S + k_t v_t^T; h0 fp32
    [N, H_v, d_k, d_v] or None. With ``cu_seqlens`` (int32 [N + 1]
    on the device) B must be 1 and the N sequences are packed along T. ``o`` and ``ht``
    may be given to write into existing buffers. ``ht`` is None in the result when
    ``output_final_state`` is False. ``one_cta_per_unit`` sets KDA_FLAG_ONE_CTA_PER_UNIT
    (never the persistent kernel that occupies every SM). ``recurrent`` computes token by
    token (kda_recurrent_fwd_ex: the decode step; ``ht`` may then be ``h0`` itself).

    Front-end (kda_chunk_fwd_fused / kda_recurrent_fwd_fused): ``qk_l2norm`` normalises q
    and k per token and head in the kernel (eps 1e-6 inside the square root);
    ``beta_sigmoid`` takes ``beta`` as logits; ``A_log`` (fp32 [H_v]) takes ``g`` as the
    gate pre-activation a and uses g = -exp(A_log) * softplus(a + dt_bias), with
    ``dt_bias`` fp32 [H_v] (per-head gate) or [H_v, d_k] (per-channel) or None.
    ``unfused_frontend`` runs the front-end as a separate pass (for comparison).
    """
    import torch

    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4:
        raise ValueError("q, k must be [B, T, H_k, d_k] and v [B, T, H_v, d_v]")
    B, T, H_k, d_k = q.shape
    _, _, H_v, d_v = v.shape
    if v.shape[:2] != (B, T):
        raise ValueError("v must share B and T with q")
    if q.dtype == torch.bfloat16:
        dtype = KDA_DTYPE_BF16
    elif q.dtype == torch.float32:
        dtype = KDA_DTYPE_F32
    else:
        raise TypeError("q, k, v must be bf16 or fp32")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if g.dtype != torch.float32 or (beta is not None and beta.dtype != torch.float32):
        raise TypeError("g and beta must be fp32")
    if g.shape == (B, T, H_v, d_k):
        gate = KDA_GATE_PER_CHANNEL
    elif g.shape == (B, T, H_v):
        gate = KDA_GATE_PER_HEAD
    else:
        raise ValueError("g must be [B, T, H_v, d_k] or [B, T, H_v]")
    if beta is not None and beta.shape != (B, T, H_v):
        raise ValueError("beta must be [B, T, H_v] (or None: the decay-only recurrence)")
    if dt_bias is not None and A_log is None:
        raise ValueError("dt_bias needs A_log")
    if A_log is not None:
        if A_log.dtype != torch.float32 or tuple(A_log.shape) != (H_v,):
            raise ValueError("A_log must be fp32 [H_v]")
        want = (H_v, d_k) if gate == KDA_GATE_PER_CHANNEL else (H_v,)
        if dt_bias is not None and (dt_bias.dtype != torch.float32 or tuple(dt_bias.shape) != want):
            raise ValueError(f"dt_bias must be fp32 {list(want)}")
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("packed sequences need B == 1")
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
            raise TypeError("cu_seqlens must be int32 [N + 1]")
        N = cu_seqlens.numel() - 1
        nb, nt = N, T
    else:
        N = B
        nb, nt = B, T
    if h0 is not None and (h0.dtype != torch.float32 or tuple(h0.shape) != (N, H_v, d_k, d_v)):
        raise ValueError("h0 must be fp32 [N, H_v, d_k, d_v]")
    # caller-provided outputs: the kernels write every element of the documented shape
    if o is not None and (o.dtype != q.dtype or tuple(o.shape) != (B, T, H_v, d_v)):
        raise ValueError("o must be [B, T, H_v, d_v] in the dtype of q")
    if ht is not None and output_final_state and (ht.dtype != torch.float32 or tuple(ht.shape) != (N, H_v, d_k, d_v)):
        raise ValueError("ht must be fp32 [N, H_v, d_k, d_v]")
    for t in (q, k, v, g, beta, h0, cu_seqlens, A_log, dt_bias, o, ht if output_final_state else None):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("every tensor must be a contiguous CUDA tensor")
    if o is None:
        o = torch.empty((B, T, H_v, d_v), dtype=q.dtype, device=q.device)
    if output_final_state and ht is None:
        ht = torch.empty((N, H_v, d_k, d_v), dtype=torch.float32, device=q.device)
    if not output_final_state:
        ht = None
    if scale is None:
        scale = d_k ** -0.5
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    p = kda_fwd_params(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta) or None, _ptr(h0) or None, _ptr(o),
                       _ptr(ht) or None, nb, nt, H_k, H_v, d_k, d_v, chunk_size, float(scale),
                       _ptr(cu_seqlens) or None, dtype, gate,
                       (KDA_FLAG_ONE_CTA_PER_UNIT if one_cta_per_unit else 0)
                       | (KDA_FLAG_UNFUSED_FRONTEND if unfused_frontend else 0))
    fused = qk_l2norm or beta_sigmoid or A_log is not None
    if recurrent:
        p.flags &= ~KDA_FLAG_ONE_CTA_PER_UNIT
    if fused:
        fe = kda_frontend(1 if qk_l2norm else 0, 1 if beta_sigmoid else 0, _ptr(A_log) or None,
                          _ptr(dt_bias) or None)
        name = "kda_recurrent_fwd_fused" if recurrent else "kda_chunk_fwd_fused"
        st = (kda_recurrent_fwd_fused if recurrent else kda_chunk_fwd_fused)(p, fe, stream)
    else:
        name = "kda_recurrent_fwd_ex" if recurrent else "kda_chunk_fwd_ex"
        st = (kda_recurrent_fwd_ex if recurrent else kda_chunk_fwd_ex)(p, stream)
    if st != KDA_OK:
        raise KdaError(st, name)
    return o, ht


def chunk_kda_bwd(q, k, v, g, beta, do, *, h0=None, dht=None, scale=None, cu_seqlens=None,
                  chunk_size=64, want_dh0=True, stream=None):
    """Backward of :func:`chunk_kda_fwd` on torch CUDA tensors (kda_chunk_bwd).

    Same inputs as the forward plus ``do`` (the gradient of o, like v) and ``dht`` (of ht,
    fp32 [N, H_v, d_k, d_v], or None). Returns ``(dq, dk, dv, dg, dbeta, dh0)``: dq, dk, dv
    in the dtype of q, dg like g, dbeta like beta (None without beta), dh0 fp32 (None when
    ``want_dh0`` is False).
    """
    import torch

    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or do.shape != v.shape:
        raise ValueError("q, k must be [B, T, H_k, d_k]; v and do [B, T, H_v, d_v]")
    B, T, H_k, d_k = q.shape
    _, _, H_v, d_v = v.shape
    if v.shape[:2] != (B, T):
        raise ValueError("v and do must share B and T with q")
    if q.dtype == torch.bfloat16:
        dtype = KDA_DTYPE_BF16
    elif q.dtype == torch.float32:
        dtype = KDA_DTYPE_F32
    else:
        raise TypeError("q, k, v must be bf16 or fp32")
    if k.dtype != q.dtype or v.dtype != q.dtype or do.dtype != q.dtype:
        raise TypeError("q, k, v and do must share one dtype")
    if g.dtype != torch.float32 or (beta is not None and beta.dtype != torch.float32):
        raise TypeError("g and beta must be fp32")
    if g.shape == (B, T, H_v, d_k):
        gate = KDA_GATE_PER_CHANNEL
    elif g.shape == (B, T, H_v):
        gate = KDA_GATE_PER_HEAD
    else:
        raise ValueError("g must be [B, T, H_v, d_k] or [B, T, H_v]")
    if beta is not None and beta.shape != (B, T, H_v):
        raise ValueError("beta must be [B, T, H_v] (or None: the decay-only recurrence)")
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("packed sequences need B == 1")
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
            raise TypeError("cu_seqlens must be int32 [N + 1]")
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    nb = N
    for name, t in (("h0", h0), ("dht", dht)):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (N, H_v, d_k, d_v)):
            raise ValueError(f"{name} must be fp32 [N, H_v, d_k, d_v]")
    for t in (q, k, v, g, beta, do, h0, dht, cu_seqlens):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("every tensor must be a contiguous CUDA tensor")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty_like(g)
    dbeta = None if beta is None else torch.empty_like(beta)
    dh0 = torch.empty((N, H_v, d_k, d_v), dtype=torch.float32, device=q.device) if want_dh0 else None
    if scale is None:
        scale = d_k ** -0.5
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    p = kda_bwd_params(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta) or None, _ptr(h0) or None,
                       _ptr(do), _ptr(dht) or None, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                       _ptr(dbeta) or None, _ptr(dh0) or None, nb, T, H_k, H_v, d_k, d_v, chunk_size,
                       float(scale), _ptr(cu_seqlens) or None, dtype, gate, 0)
    st = kda_chunk_bwd(p, stream)
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_bwd")
    return dq, dk, dv, dg, dbeta, dh0
