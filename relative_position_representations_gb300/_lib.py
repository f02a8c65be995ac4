"""ctypes binding of librelattn.so — argument marshalling only.

Each function has the name of the C entry point it calls (include/relattn.h). Tensors are
torch CUDA tensors (torch is used for device memory and streams only): the binding checks
device, dtype, shape and contiguity, passes raw pointers and the current CUDA stream, and
raises RelattnError on a non-OK status. Every step of the computation runs in the
library's kernels; if the library is missing this module raises at import time.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librelattn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
BF16, F32 = 0, 1

if not os.path.exists(LIB_PATH):
    raise ImportError("librelattn.so is not built (%s); run `python -c \"import __graft_entry__ "
                      "as g; g.build()\"` first" % LIB_PATH)
_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_lib.relattn_fwd.argtypes = [_P, _P, _P, _P, _P, ctypes.c_longlong, _I, _I, ctypes.c_float, _P,
                             _I, _I, _I, _I, _I, _P, _P]
_lib.relattn_fwd.restype = _I
_lib.relattn_t5bias_fwd.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P, _I, _I,
                                    _I, _I, _I, _P, _P]
_lib.relattn_t5bias_fwd.restype = _I
_lib.relattn_alibi_fwd.argtypes = [_P, _P, _P, _P, _I, ctypes.c_float, _P, _I, _I, _I, _I, _I,
                                   _P, _P]
_lib.relattn_alibi_fwd.restype = _I
_lib.relattn_offset_bias_fwd.argtypes = [_P, _P, _P, _P, ctypes.c_longlong, _I, _I,
                                         ctypes.c_float, _P, _I, _I, _I, _I, _I, _P, _P]
_lib.relattn_offset_bias_fwd.restype = _I
_lib.relattn_labeled_fwd.argtypes = [_P, _P, _P, _P, _P, ctypes.c_longlong, _I, _P,
                                     ctypes.c_longlong, _I, ctypes.c_float, _P, _I, _I, _I, _I,
                                     _I, _P, _P]
_lib.relattn_labeled_fwd.restype = _I
_lib.relattn_txl_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, ctypes.c_float, _P, _I, _I, _I,
                                 _I, _I, _P, _P]
_lib.relattn_txl_fwd.restype = _I
_lib.relattn_decode_fwd.argtypes = [_P, _P, _P, _P, _P, ctypes.c_longlong, _I, ctypes.c_float, _P,
                                    _I, _I, _I, _I, _P, ctypes.c_ulonglong, _P, _P]
_lib.relattn_decode_fwd.restype = _I
_lib.relattn_decode_fwd_noalloc.argtypes = [_P, _P, _P, _P, _P, ctypes.c_longlong, _I,
                                            ctypes.c_float, _P, _I, _I, _I, _I, _P, _P]
_lib.relattn_decode_fwd_noalloc.restype = _I
_lib.relattn_bwd.argtypes = [_P, _P, _P, _P, _P, ctypes.c_longlong, _I, _I, ctypes.c_float, _P, _I,
                             _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_ulonglong, _P]
_lib.relattn_bwd.restype = _I
_lib.relattn_bwd_workspace_size.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_ulonglong)]
_lib.relattn_bwd_workspace_size.restype = _I
_lib.relattn_scalar_bias_bwd.argtypes = [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, ctypes.c_longlong,
                                         _I, ctypes.c_float, _P, _I, _I, _I, _I, _I, _P, _P, _P,
                                         _P, _P, ctypes.c_ulonglong, _P]
_lib.relattn_scalar_bias_bwd.restype = _I
_lib.relattn_scalar_bias_bwd_workspace_size.argtypes = [_I, _I, _I, ctypes.POINTER(ctypes.c_ulonglong)]
_lib.relattn_scalar_bias_bwd_workspace_size.restype = _I
_lib.relattn_labeled_bwd.argtypes = [_P, _P, _P, _P, _P, ctypes.c_longlong, _I, _P,
                                     ctypes.c_longlong, _I, ctypes.c_float, _P, _I, _I, _I, _I,
                                     _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_ulonglong, _P]
_lib.relattn_labeled_bwd.restype = _I
_lib.relattn_labeled_bwd_workspace_size.argtypes = [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_ulonglong)]
_lib.relattn_labeled_bwd_workspace_size.restype = _I
_lib.relattn_decode_workspace_size.argtypes = [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_ulonglong)]
_lib.relattn_decode_workspace_size.restype = _I
_lib.relattn_labels.argtypes = [_I, _I, _I, _I, _I, _I, _I, _P, _P]
_lib.relattn_labels.restype = _I
_lib.relattn_t5_thresholds.argtypes = [_I, _I, _I, ctypes.POINTER(_I), _I, ctypes.POINTER(_I)]
_lib.relattn_t5_thresholds.restype = _I
_lib.relattn_get_device_error.argtypes = [_P]
_lib.relattn_get_device_error.restype = _I
_lib.relattn_status_string.argtypes = [_I]
_lib.relattn_status_string.restype = ctypes.c_char_p
_lib.relattn_set_wait_limit.argtypes = [ctypes.c_longlong]
_lib.relattn_set_wait_limit.restype = _I
_lib.relattn_debug_withhold_first_load.argtypes = [_I]
_lib.relattn_debug_withhold_first_load.restype = _I
_lib.relattn_set_short_kernel.argtypes = [_I]
_lib.relattn_set_short_kernel.restype = _I
_lib.relattn_sinusoid_table.argtypes = [_I, _I, _I, _P, _P]
_lib.relattn_sinusoid_table.restype = _I
_lib.relattn_set_bwd_tensor_cores.argtypes = [_I]
_lib.relattn_set_bwd_tensor_cores.restype = _I
_lib.relattn_version.argtypes = []
_lib.relattn_version.restype = _I

EXPORTED = ["relattn_fwd", "relattn_t5bias_fwd", "relattn_alibi_fwd",
            "relattn_offset_bias_fwd", "relattn_labeled_fwd", "relattn_txl_fwd", "relattn_sinusoid_table",
            "relattn_decode_fwd",
            "relattn_decode_fwd_noalloc", "relattn_decode_workspace_size", "relattn_bwd",
            "relattn_bwd_workspace_size", "relattn_scalar_bias_bwd",
            "relattn_scalar_bias_bwd_workspace_size", "relattn_labeled_bwd",
            "relattn_labeled_bwd_workspace_size", "relattn_labels",
            "relattn_t5_thresholds", "relattn_set_wait_limit",
            "relattn_debug_withhold_first_load", "relattn_set_short_kernel", "relattn_set_bwd_tensor_cores",
            "relattn_get_device_error", "relattn_status_string", "relattn_version"]


class RelattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, relattn_status_string(status), status))


def relattn_status_string(status: int) -> str:
    return _lib.relattn_status_string(int(status)).decode()


def relattn_version() -> int:
    return int(_lib.relattn_version())


def _check(status: int, where: str):
    if status != OK:
        raise RelattnError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name, q.dtype)
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError("%s must be [B, H, n, d] like q" % name)
    return q.shape


def relattn_fwd(q, k, v, aK=None, aV=None, clip_k=0, causal=False, scale=None, kv_len=None,
                out=None, table_head_stride=None, stream=None):
    """Shaw relation-aware attention forward ("Self-Attention with Relative Position Representations"
    page, section 3.4, eqs. 3-4).

    q, k, v: [B, H, n, d] bf16 or fp32 CUDA tensors. aK / aV: [H or 1, 2*clip_k+1, d]
    (None drops the term). kv_len: [B] int32 CUDA tensor or None. Returns out.
    """
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    W = 2 * int(clip_k) + 1
    for name, t in (("aK", aK), ("aV", aV)):
        if t is not None:
            _dev(t, name, q.dtype)
            if t.dim() != 3 or t.shape[1] != W or t.shape[2] != d or t.shape[0] not in (1, H):
                raise ValueError("%s must be [H or 1, 2*clip_k+1, d]" % name)
    if table_head_stride is None:
        ref = aK if aK is not None else aV
        table_head_stride = 0 if (ref is None or ref.shape[0] == 1) else W * d
    _dev(kv_len, "kv_len", torch.int32)
    if kv_len is not None and kv_len.numel() != B:
        raise ValueError("kv_len must have B entries")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    if scale is None:
        scale = d ** -0.5
    st = _lib.relattn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(aK), _ptr(aV), int(table_head_stride),
                          int(clip_k), int(bool(causal)), float(scale), _ptr(kv_len), B, H, n, d,
                          dt, _ptr(out), _stream(stream))
    _check(st, "relattn_fwd")
    return out


def relattn_t5bias_fwd(q, k, v, bias, num_buckets=32, max_distance=128, bidirectional=True,
                       causal=False, scale=1.0, kv_len=None, out=None, stream=None):
    """T5 scalar bucketed-bias attention ("Relative position embeddings", section "T5").

    bias: [num_buckets, H] fp32 CUDA tensor. Returns out.
    """
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    _dev(bias, "bias", torch.float32)
    if bias.shape != (num_buckets, H):
        raise ValueError("bias must be [num_buckets, H]")
    _dev(kv_len, "kv_len", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    st = _lib.relattn_t5bias_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), int(num_buckets),
                                 int(max_distance), int(bool(bidirectional)), int(bool(causal)),
                                 float(scale), _ptr(kv_len), B, H, n, d, dt, _ptr(out),
                                 _stream(stream))
    _check(st, "relattn_t5bias_fwd")
    return out


def relattn_alibi_fwd(q, k, v, slopes, causal=False, scale=None, kv_len=None, out=None,
                      stream=None):
    """ALiBi attention: e_ij = scale * q_i . k_j - slopes[h] * |j - i| ("Relative position
    embeddings", section "Placement in the taxonomy").

    slopes: [H] fp32 CUDA tensor. scale defaults to 1/sqrt(d). Returns out.
    """
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    _dev(slopes, "slopes", torch.float32)
    if slopes.shape != (H,):
        raise ValueError("slopes must be [H]")
    _dev(kv_len, "kv_len", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    if scale is None:
        scale = d ** -0.5
    st = _lib.relattn_alibi_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(slopes), int(bool(causal)),
                                float(scale), _ptr(kv_len), B, H, n, d, dt, _ptr(out),
                                _stream(stream))
    _check(st, "relattn_alibi_fwd")
    return out


def relattn_offset_bias_fwd(q, k, v, table, radius, causal=False, scale=None, kv_len=None,
                            out=None, stream=None):
    """Scalar bias per relative offset, clipped at `radius`: e_ij = scale * q_i . k_j +
    table[h, clip(j - i, radius) + radius].

    table: [H or 1, 2*radius + 1] fp32 CUDA tensor (one row: shared by every head).
    scale defaults to 1/sqrt(d). Returns out.
    """
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    _dev(table, "table", torch.float32)
    W = 2 * int(radius) + 1
    if table.dim() != 2 or table.shape[1] != W or table.shape[0] not in (1, H):
        raise ValueError("table must be [H or 1, 2*radius + 1]")
    ths = 0 if (table.shape[0] == 1 and H > 1) else W
    _dev(kv_len, "kv_len", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    if scale is None:
        scale = d ** -0.5
    st = _lib.relattn_offset_bias_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(table), int(ths),
                                      int(radius), int(bool(causal)), float(scale),
                                      _ptr(kv_len), B, H, n, d, dt, _ptr(out), _stream(stream))
    _check(st, "relattn_offset_bias_fwd")
    return out


def relattn_txl_fwd(q, k, v, rel, u, vb, causal=False, scale=None, kv_len=None, out=None,
                    stream=None):
    """Transformer-XL relative attention: score (q_i + u) . k_j + (q_i + v) . rel[j - i + n - 1]
    ("Relative Position Encoding in Transformer-XL" page, the four-term score).

    rel: [H or 1, 2n - 1, d], u and vb: [H or 1, d], all of q's dtype (one set for every head
    when the first dimension is 1 and H > 1). scale defaults to 1/sqrt(d). Returns out.
    """
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    for t, nm in ((rel, "rel"), (u, "u"), (vb, "vb")):
        _dev(t, nm, q.dtype)
    if rel.dim() != 3 or rel.shape[1:] != (2 * n - 1, d) or u.dim() != 2 or vb.dim() != 2:
        raise ValueError("rel must be [H or 1, 2n - 1, d], u and vb [H or 1, d]")
    shared = 1 if (rel.shape[0] == 1 and H > 1) else 0
    if rel.shape[0] != (1 if shared else H) or u.shape != (rel.shape[0], d) or vb.shape != u.shape:
        raise ValueError("rel, u and vb must have one entry per head, or one for all")
    _dev(kv_len, "kv_len", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    if scale is None:
        scale = d ** -0.5
    st = _lib.relattn_txl_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(rel), _ptr(u), _ptr(vb), shared,
                              int(bool(causal)), float(scale), _ptr(kv_len), B, H, n, d, dt,
                              _ptr(out), _stream(stream))
    _check(st, "relattn_txl_fwd")
    return out


def relattn_labeled_fwd(q, k, v, labels, aK=None, aV=None, causal=False, scale=None,
                        kv_len=None, out=None, table_head_stride=None, stream=None):
    """Relation-aware attention over labelled edges: the table rows of edge (i, j) are picked
    by labels[b, i, j] ("Self-Attention with Relative Position Representations" page, section
    "Relation-Aware Self-Attention: The Core Modification").

    labels: uint8 CUDA tensor [n, n] (shared by every sequence) or [B, n, n]. aK / aV:
    [H or 1, num_labels, d] of q's dtype, or None. scale defaults to 1/sqrt(d). Returns out.
    """
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    ref = aK if aK is not None else aV
    num_labels = 0
    lbs = 0
    if ref is not None:
        for t, nm in ((aK, "aK"), (aV, "aV")):
            _dev(t, nm, q.dtype)
        if ref.dim() != 3 or ref.shape[2] != d:
            raise ValueError("tables must be [H or 1, num_labels, d]")
        num_labels = int(ref.shape[1])
        if table_head_stride is None:
            table_head_stride = 0 if (ref.shape[0] == 1 and H > 1) else num_labels * d
        _dev(labels, "labels", torch.uint8)
        if labels.shape == (n, n):
            lbs = 0
        elif labels.shape == (B, n, n):
            lbs = n * n
        else:
            raise ValueError("labels must be [n, n] or [B, n, n]")
    else:
        table_head_stride = 0
    _dev(kv_len, "kv_len", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    if scale is None:
        scale = d ** -0.5
    st = _lib.relattn_labeled_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(aK), _ptr(aV),
                                  int(table_head_stride), num_labels,
                                  _ptr(labels) if ref is not None else None, int(lbs),
                                  int(bool(causal)), float(scale), _ptr(kv_len), B, H, n, d, dt,
                                  _ptr(out), _stream(stream))
    _check(st, "relattn_labeled_fwd")
    return out


def relattn_decode_fwd_noalloc(q, k_cache, v_cache, cache_len, aK=None, aV=None, clip_k=0,
                               scale=None, out=None, table_head_stride=None, stream=None):
    """relattn_decode_fwd with the library's built-in device scratch (no workspace argument;
    calls on different streams must not overlap). Same arguments and result."""
    B, H, d = q.shape
    T = k_cache.shape[2]
    W = 2 * int(clip_k) + 1
    if table_head_stride is None:
        ref = aK if aK is not None else aV
        table_head_stride = 0 if (ref is None or ref.shape[0] == 1) else W * d
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.bfloat16)
    if scale is None:
        scale = d ** -0.5
    st = _lib.relattn_decode_fwd_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(aK),
                                         _ptr(aV), int(table_head_stride), int(clip_k),
                                         float(scale), _ptr(cache_len), B, H, T, d, _ptr(out),
                                         _stream(stream))
    _check(st, "relattn_decode_fwd_noalloc")
    return out


def relattn_bwd_workspace_size(B, H, n, d, clip_k) -> int:
    """Workspace bytes relattn_bwd needs (host only)."""
    nb = ctypes.c_ulonglong(0)
    _check(_lib.relattn_bwd_workspace_size(int(B), int(H), int(n), int(d), int(clip_k),
                                           ctypes.byref(nb)), "relattn_bwd_workspace_size")
    return int(nb.value)


def relattn_bwd(q, k, v, dout, aK=None, aV=None, clip_k=0, causal=False, scale=None, kv_len=None,
                table_head_stride=None, workspace=None, stream=None):
    """Gradients of relattn_fwd: returns (dq, dk, dv, daK, daV), fp32 (daK / daV None when
    the table is None). workspace: a CUDA tensor of at least relattn_bwd_workspace_size
    bytes, or None to make one."""
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    _dev(dout, "dout", q.dtype)
    if dout.shape != q.shape:
        raise ValueError("dout must be [B, H, n, d] like q")
    W = 2 * int(clip_k) + 1
    for name, t in (("aK", aK), ("aV", aV)):
        if t is not None:
            _dev(t, name, q.dtype)
            if t.dim() != 3 or t.shape[1] != W or t.shape[2] != d or t.shape[0] not in (1, H):
                raise ValueError("%s must be [H or 1, 2*clip_k+1, d]" % name)
    if table_head_stride is None:
        ref = aK if aK is not None else aV
        table_head_stride = 0 if (ref is None or ref.shape[0] == 1) else W * d
    _dev(kv_len, "kv_len", torch.int32)
    if scale is None:
        scale = d ** -0.5
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dv = (torch.empty(q.shape, **f32) for _ in range(3))
    daK = None if aK is None else torch.empty(aK.shape, **f32)
    daV = None if aV is None else torch.empty(aV.shape, **f32)
    need = relattn_bwd_workspace_size(B, H, n, d, clip_k)
    if workspace is None:
        workspace = torch.empty(max(need, 4), dtype=torch.uint8, device=q.device)
    _dev(workspace, "workspace")
    st = _lib.relattn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(aK), _ptr(aV), int(table_head_stride),
                          int(clip_k), int(bool(causal)), float(scale), _ptr(kv_len), B, H, n, d,
                          dt, _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(daK), _ptr(daV),
                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream(stream))
    _check(st, "relattn_bwd")
    return dq, dk, dv, daK, daV


def relattn_scalar_bias_bwd_workspace_size(B, H, n) -> int:
    """Workspace bytes relattn_scalar_bias_bwd needs (host only)."""
    nb = ctypes.c_ulonglong(0)
    _check(_lib.relattn_scalar_bias_bwd_workspace_size(int(B), int(H), int(n), ctypes.byref(nb)),
           "relattn_scalar_bias_bwd_workspace_size")
    return int(nb.value)


_BIAS_KINDS = {"t5": 0, "alibi": 1, "table": 2}


def relattn_scalar_bias_bwd(q, k, v, dout, kind, bias, num_buckets=32, max_distance=128,
                            bidirectional=True, radius=0, causal=False, scale=None, kv_len=None,
                            workspace=None, stream=None):
    """Gradients of the scalar offset-bias forwards: returns (dq, dk, dv, dbias), fp32.

    kind "t5": bias [num_buckets, H] (relattn_t5bias_fwd; scale defaults to 1.0);
    "alibi": slopes [H] (relattn_alibi_fwd); "table": [H or 1, 2*radius+1]
    (relattn_offset_bias_fwd; one row is shared by the heads). dbias has bias's shape.
    workspace: a CUDA tensor of at least relattn_scalar_bias_bwd_workspace_size bytes, or
    None to make one."""
    if kind not in _BIAS_KINDS:
        raise ValueError("kind must be one of %s" % sorted(_BIAS_KINDS))
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    _dev(dout, "dout", q.dtype)
    if dout.shape != q.shape:
        raise ValueError("dout must be [B, H, n, d] like q")
    if bias is None:
        raise ValueError("bias is required")
    _dev(bias, "bias", torch.float32)
    hs = 0
    if kind == "t5":
        if bias.shape != (int(num_buckets), H):
            raise ValueError("bias must be [num_buckets, H]")
    elif kind == "alibi":
        if bias.shape != (H,):
            raise ValueError("slopes must be [H]")
    else:
        W = 2 * int(radius) + 1
        if bias.dim() != 2 or bias.shape[1] != W or bias.shape[0] not in (1, H):
            raise ValueError("table must be [H or 1, 2*radius+1]")
        hs = 0 if bias.shape[0] == 1 else W
    _dev(kv_len, "kv_len", torch.int32)
    if scale is None:
        scale = 1.0 if kind == "t5" else d ** -0.5
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dv = (torch.empty(q.shape, **f32) for _ in range(3))
    dbias = torch.empty(bias.shape, **f32)
    need = relattn_scalar_bias_bwd_workspace_size(B, H, n)
    if workspace is None:
        workspace = torch.empty(max(need, 4), dtype=torch.uint8, device=q.device)
    _dev(workspace, "workspace")
    st = _lib.relattn_scalar_bias_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _BIAS_KINDS[kind], _ptr(bias), int(num_buckets),
        int(max_distance), int(bool(bidirectional)), int(radius), hs, int(bool(causal)),
        float(scale), _ptr(kv_len), B, H, n, d, dt, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "relattn_scalar_bias_bwd")
    return dq, dk, dv, dbias


def relattn_labeled_bwd_workspace_size(B, H, n, num_labels) -> int:
    """Workspace bytes relattn_labeled_bwd needs (host only)."""
    nb = ctypes.c_ulonglong(0)
    _check(_lib.relattn_labeled_bwd_workspace_size(int(B), int(H), int(n), int(num_labels),
                                                   ctypes.byref(nb)),
           "relattn_labeled_bwd_workspace_size")
    return int(nb.value)


def relattn_labeled_bwd(q, k, v, dout, labels, aK=None, aV=None, num_labels=None, causal=False,
                        scale=None, kv_len=None, table_head_stride=None, workspace=None,
                        stream=None):
    """Gradients of relattn_labeled_fwd: returns (dq, dk, dv, daK, daV), fp32 (daK / daV None
    when the table is None). labels: uint8 [n, n] or [B, n, n]; num_labels defaults to the
    tables' row count (required without tables). workspace: a CUDA tensor of at least
    relattn_labeled_bwd_workspace_size bytes, or None to make one."""
    B, H, n, d = _qkv(q, k, v)
    dt = _dtype_code(q)
    _dev(dout, "dout", q.dtype)
    if dout.shape != q.shape:
        raise ValueError("dout must be [B, H, n, d] like q")
    ref = aK if aK is not None else aV
    for t, nm in ((aK, "aK"), (aV, "aV")):
        if t is not None:
            _dev(t, nm, q.dtype)
            if t.dim() != 3 or t.shape[2] != d or t.shape[0] not in (1, H):
                raise ValueError("tables must be [H or 1, num_labels, d]")
    if num_labels is None:
        if ref is None:
            raise ValueError("num_labels is required without tables")
        num_labels = int(ref.shape[1])
    if table_head_stride is None:
        table_head_stride = 0 if (ref is None or ref.shape[0] == 1) else int(num_labels) * d
    _dev(labels, "labels", torch.uint8)
    if labels is None:
        raise ValueError("labels is required")
    if labels.shape == (n, n):
        lbs = 0
    elif labels.shape == (B, n, n):
        lbs = n * n
    else:
        raise ValueError("labels must be [n, n] or [B, n, n]")
    _dev(kv_len, "kv_len", torch.int32)
    if scale is None:
        scale = d ** -0.5
    f32 = dict(dtype=torch.float32, device=q.device)
    dq, dk, dv = (torch.empty(q.shape, **f32) for _ in range(3))
    daK = None if aK is None else torch.empty(aK.shape, **f32)
    daV = None if aV is None else torch.empty(aV.shape, **f32)
    need = relattn_labeled_bwd_workspace_size(B, H, n, num_labels)
    if workspace is None:
        workspace = torch.empty(max(need, 4), dtype=torch.uint8, device=q.device)
    _dev(workspace, "workspace")
    st = _lib.relattn_labeled_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(aK), _ptr(aV),
                                  int(table_head_stride), int(num_labels), _ptr(labels), int(lbs),
                                  int(bool(causal)), float(scale), _ptr(kv_len), B, H, n, d, dt,
                                  _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(daK), _ptr(daV),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check(st, "relattn_labeled_bwd")
    return dq, dk, dv, daK, daV


def relattn_decode_workspace_size(B, H, T, d) -> int:
    """Workspace bytes relattn_decode_fwd uses to split all caches over the GPU (host only)."""
    n = ctypes.c_ulonglong(0)
    _check(_lib.relattn_decode_workspace_size(int(B), int(H), int(T), int(d), ctypes.byref(n)),
           "relattn_decode_workspace_size")
    return int(n.value)


def relattn_decode_fwd(q, k_cache, v_cache, cache_len, aK=None, aV=None, clip_k=0, scale=None,
                       out=None, table_head_stride=None, workspace=None, stream=None):
    """One causal decoding step with relative terms: row cache_len[b] - 1 of the causal
    forward over each sequence's cache ("Self-Attention with Relative Position Representations"
    page, section 3.4, eqs. 3-4).

    q: [B, H, d] bf16; k_cache, v_cache: [B, H, T, d] bf16; cache_len: [B] int32 (the new
    token's key and value already in row cache_len[b] - 1). aK / aV: [H or 1, 2*clip_k+1, d]
    bf16 or None. workspace: a CUDA tensor of at least relattn_decode_workspace_size bytes
    (None: one CTA per cache). Returns out [B, H, d].
    """
    _dev(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [B, H, d]")
    B, H, d = q.shape
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, name, torch.bfloat16)
        if t.dim() != 4 or t.shape[0] != B or t.shape[1] != H or t.shape[3] != d:
            raise ValueError("%s must be [B, H, T, d]" % name)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must have one shape")
    T = k_cache.shape[2]
    W = 2 * int(clip_k) + 1
    for name, t in (("aK", aK), ("aV", aV)):
        if t is not None:
            _dev(t, name, torch.bfloat16)
            if t.dim() != 3 or t.shape[1] != W or t.shape[2] != d or t.shape[0] not in (1, H):
                raise ValueError("%s must be [H or 1, 2*clip_k+1, d]" % name)
    if table_head_stride is None:
        ref = aK if aK is not None else aV
        table_head_stride = 0 if (ref is None or ref.shape[0] == 1) else W * d
    _dev(cache_len, "cache_len", torch.int32)
    if cache_len.numel() != B:
        raise ValueError("cache_len must have B entries")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.bfloat16)
    if scale is None:
        scale = d ** -0.5
    ws_bytes = 0
    if workspace is not None:
        _dev(workspace, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.relattn_decode_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(aK), _ptr(aV),
                                 int(table_head_stride), int(clip_k), float(scale),
                                 _ptr(cache_len), B, H, T, d, _ptr(workspace), ws_bytes, _ptr(out),
                                 _stream(stream))
    _check(st, "relattn_decode_fwd")
    return out


def relattn_labels(kind, n_q, n_k, clip_k=0, num_buckets=32, max_distance=128,
                   bidirectional=True, out=None, stream=None, device=None):
    """Edge label of every (i, j) from the device index functions: int32 [n_q, n_k].

    kind "clip": clip(j - i, clip_k) + clip_k. kind "t5": T5 bucket(j - i).
    """
    code = {"clip": 0, "t5": 1}[kind]
    if out is None:
        out = torch.empty((n_q, n_k), dtype=torch.int32,
                          device=device or torch.device("cuda", torch.cuda.current_device()))
    _dev(out, "out", torch.int32)
    st = _lib.relattn_labels(code, int(clip_k), int(num_buckets), int(max_distance),
                             int(bool(bidirectional)), int(n_q), int(n_k), _ptr(out),
                             _stream(stream))
    _check(st, "relattn_labels")
    return out


def relattn_t5_thresholds(num_buckets=32, max_distance=128, bidirectional=True):
    """First distance of each logarithmic T5 bucket of one half (host computation)."""
    cap = 256
    arr = (_I * cap)()
    cnt = _I(0)
    st = _lib.relattn_t5_thresholds(int(num_buckets), int(max_distance), int(bool(bidirectional)),
                                    arr, cap, ctypes.byref(cnt))
    _check(st, "relattn_t5_thresholds")
    return [arr[i] for i in range(cnt.value)]


def relattn_get_device_error(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(_lib.relattn_get_device_error(_stream(stream)))


def relattn_set_wait_limit(cycles: int) -> None:
    """Bound of every device wait of the tensor-core forward kernels, in SM clock cycles."""
    st = int(_lib.relattn_set_wait_limit(int(cycles)))
    if st != OK:
        raise RelattnError(st, "relattn_set_wait_limit")


def relattn_debug_withhold_first_load(on: bool) -> None:
    """Test hook: the tensor-core forward kernels withhold their first Q load (timeout test)."""
    st = int(_lib.relattn_debug_withhold_first_load(1 if on else 0))
    if st != OK:
        raise RelattnError(st, "relattn_debug_withhold_first_load")


def relattn_set_short_kernel(on: bool) -> None:
    """Route bf16 forwards of at most 256 keys with d = 64 to the short-sequence kernel (default)."""
    st = int(_lib.relattn_set_short_kernel(1 if on else 0))
    if st != OK:
        raise RelattnError(st, "relattn_set_short_kernel")


def relattn_sinusoid_table(n, d_model, dtype=None, device=None, stream=None):
    """The sinusoidal encodings of the offsets -(n-1) .. n-1: a [2n - 1, d_model] tensor
    (bf16 by default) on `device` (default the current CUDA device)."""
    dtype = torch.bfloat16 if dtype is None else dtype
    out = torch.empty((2 * int(n) - 1, int(d_model)), dtype=dtype,
                      device=device if device is not None else "cuda")
    st = _lib.relattn_sinusoid_table(int(n), int(d_model), _dtype_code(out), _ptr(out), _stream(stream))
    _check(st, "relattn_sinusoid_table")
    return out


def relattn_set_bwd_tensor_cores(on: bool) -> None:
    """Route eligible bf16 gradient calls to the tensor-core kernels (default) or the SIMT ones."""
    st = int(_lib.relattn_set_bwd_tensor_cores(1 if on else 0))
    if st != OK:
        raise RelattnError(st, "relattn_set_bwd_tensor_cores")


def raw_call(name, *args):
    """Call an exported C function directly with ctypes arguments (tests of the ABI)."""
    return getattr(_lib, name)(*args)
