"""fp64 CPU oracle for relation-aware self-attention and the T5 bucketed bias.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference leg may import this package. The CUDA library never loads it, and
it shares no code with the CUDA library: the compute loop is plain C in
relattn_oracle.c (built with gcc, no fast-math), the exact T5 bucketing is oracle/t5.py,
and a second, numpy-only statement of the same formulas (materialised edge tensors and
the split form) lives in oracle/brute.py.

Every function takes numpy arrays (any float dtype; they are widened to float64 here,
which is exact for bf16 and fp32 inputs) and returns float64 results.

Pins (tests/test_oracle_pins.py): reduction to library scaled-dot-product attention when
the tables are zero, the k = 0 closed forms, the causal first row, shift invariance of
the relative-only dependence, the brute-force materialised form, bin sums, key-only
equivalence, T5 constant-bias reduction, the clip examples and label counts printed on
the pages, and a hand-computed 2-token sign check.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import t5 as _t5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "relattn_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile relattn_oracle.c into oracle/liboracle.so with gcc (IEEE fp64, no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _configure(lib):
    P = ctypes.c_void_p
    lib.oracle_relattn_rows.argtypes = [P, P, P, P, P, ctypes.c_longlong, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_double, P,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, P, ctypes.c_longlong, P, ctypes.c_int]
    lib.oracle_relattn_rows.restype = ctypes.c_int
    lib.oracle_t5bias_rows.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_double, P,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, P, ctypes.c_longlong, P, ctypes.c_int]
    lib.oracle_t5bias_rows.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows_arg(rows, B, H, n):
    if rows is None:
        return None, B * H * n
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    if r.size and (r.min() < 0 or r.max() >= B * H * n):
        raise ValueError("row id out of range")
    return r, int(r.size)


def clip(x, k):
    """clip(x, k) = max(-k, min(k, x)) (paper summary, "Relative Position Representations")."""
    return max(-k, min(k, x))


def relattn_fwd(q, k, v, aK, aV, clip_k, causal, scale, kv_len=None,
                table_head_stride=None, rows=None, nthreads=None):
    """Shaw relation-aware attention forward, fp64.

    q, k, v: [B, H, n, d]. aK / aV: [H_t, 2*clip_k + 1, d] or None (term absent).
    table_head_stride: elements between heads' tables (default (2k+1)*d, 0 = shared).
    rows: optional flat row ids (b*H + h)*n + i; returns [len(rows), d] then, else [B,H,n,d].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    aK, aV = _f64(aK), _f64(aV)
    if table_head_stride is None:
        table_head_stride = (2 * clip_k + 1) * d
    kvl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    r, nrows = _rows_arg(rows, B, H, n)
    out = np.zeros((nrows, d), dtype=np.float64)
    rc = _load().oracle_relattn_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(aK), _ptr(aV),
                                     int(table_head_stride), int(clip_k), int(bool(causal)),
                                     float(scale), _ptr(kvl), B, H, n, d, _ptr(r), nrows,
                                     _ptr(out), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle thread start failed")
    return out if rows is not None else out.reshape(B, H, n, d)


def t5bias_fwd(q, k, v, bias, num_buckets, max_distance, bidirectional, causal, scale,
               kv_len=None, rows=None, nthreads=None):
    """T5 scalar bucketed-bias attention forward, fp64. bias: [num_buckets, H]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    bias = _f64(bias)
    table = np.ascontiguousarray(np.asarray(
        _t5.bucket_of_offset_table(n, num_buckets, max_distance, bool(bidirectional)),
        dtype=np.int32))
    kvl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    r, nrows = _rows_arg(rows, B, H, n)
    out = np.zeros((nrows, d), dtype=np.float64)
    rc = _load().oracle_t5bias_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(table),
                                    int(bool(causal)), float(scale), _ptr(kvl), B, H, n, d,
                                    _ptr(r), nrows, _ptr(out),
                                    int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle thread start failed")
    return out if rows is not None else out.reshape(B, H, n, d)


def clip_labels(n_q: int, n_k: int, clip_k: int) -> np.ndarray:
    """Table row r = clip(j - i, k) + k for every (i, j): int32 [n_q, n_k]."""
    out = np.empty((n_q, n_k), dtype=np.int32)
    for i in range(n_q):
        for j in range(n_k):
            out[i, j] = clip(j - i, clip_k) + clip_k
    return out


def t5_labels(n_q: int, n_k: int, num_buckets: int, max_distance: int,
              bidirectional: bool) -> np.ndarray:
    """T5 bucket of (j - i) for every (i, j): int32 [n_q, n_k]."""
    cache = {}
    out = np.empty((n_q, n_k), dtype=np.int32)
    for i in range(n_q):
        for j in range(n_k):
            dl = j - i
            if dl not in cache:
                cache[dl] = _t5.t5_bucket(dl, num_buckets, max_distance, bidirectional)
            out[i, j] = cache[dl]
    return out


t5_bucket = _t5.t5_bucket
