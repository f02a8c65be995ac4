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
Pins of the scalar offset biases (ALiBi, the clipped per-offset table) are in
tests/test_oracle_offset_bias.py: library attention with the bias grid as an additive mask,
ALiBi as the T5 path with a linear table, the zero-query closed form of the ALiBi weights,
a hand-computed 2-token sign check of the clipped table, and the softmax's shift invariance.
Pins of the labelled-edge form (labeled_fwd) are in tests/test_oracle_labeled.py: clip
labels reproduce the Shaw forward, random labels match the numpy materialised form, a
2-token hand computation with asymmetric labels, constant-label closed forms, per-sequence
independence; test_oracle_mutations.py plants a transposed and a batch-blind label read.
oracle/txl.py states the Transformer-XL four-term score (pinned in tests/test_oracle_txl.py
against library attention, the Shaw loop with an unclipped table, and the offset-bias loop).
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
    lib.oracle_labeled_rows.argtypes = [P, P, P, P, P, ctypes.c_longlong, P, ctypes.c_longlong,
                                        ctypes.c_int, ctypes.c_double, P, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                        ctypes.c_longlong, P, ctypes.c_int]
    lib.oracle_labeled_rows.restype = ctypes.c_int
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
    """clip(x, k) = max(-k, min(k, x)) ("Self-Attention with Relative Position Representations" page, section "Relative Position Representations")."""
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


def labeled_fwd(q, k, v, aK, aV, labels, causal, scale, kv_len=None, table_head_stride=None,
                rows=None, nthreads=None):
    """Relation-aware attention over arbitrary labelled edges, fp64 ("Self-Attention with Relative Position Representations" page,
    section "Relation-Aware Self-Attention: The Core Modification", eqs. 3 and 4 with
    a^K_ij = w^K[L_b[i, j]] and a^V_ij = w^V[L_b[i, j]]).

    labels: uint8 [n, n] (one label matrix for every sequence) or [B, n, n]; every value
    must index a table row. aK / aV: [H_t, num_labels, d] or None. table_head_stride:
    elements between heads' tables (default num_labels * d, 0 = shared).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    aK, aV = _f64(aK), _f64(aV)
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.uint8))
    if lab.shape == (n, n):
        lbs = 0
    elif lab.shape == (B, n, n):
        lbs = n * n
    else:
        raise ValueError("labels must be [n, n] or [B, n, n]")
    ref = aK if aK is not None else aV
    if ref is not None:
        if ref.ndim != 3 or ref.shape[2] != d:
            raise ValueError("tables must be [H_t, num_labels, d]")
        if lab.size and int(lab.max()) >= ref.shape[1]:
            raise ValueError("a label has no table row")
        if table_head_stride is None:
            table_head_stride = ref.shape[1] * d
    else:
        table_head_stride = 0
    kvl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    r, nrows = _rows_arg(rows, B, H, n)
    out = np.zeros((nrows, d), dtype=np.float64)
    rc = _load().oracle_labeled_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(aK), _ptr(aV),
                                     int(table_head_stride), _ptr(lab), lbs,
                                     int(bool(causal)), float(scale), _ptr(kvl), B, H, n, d,
                                     _ptr(r), nrows, _ptr(out), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle thread start failed")
    return out if rows is not None else out.reshape(B, H, n, d)


def offset_bias_fwd(q, k, v, bias_of_offset, causal, scale, kv_len=None, rows=None,
                    nthreads=None):
    """Attention with a scalar bias per relative offset, fp64:

        e_ij = scale * q_i . k_j + bias_of_offset[h, (j - i) + n - 1]

    ("Relative position embeddings" page: the T5 form of section "T5" with the bucketing
    left out, which is what section "Placement in the taxonomy" varies). bias_of_offset:
    [H, 2n - 1], the bias of every offset of the sequence. The C loop runs it as the T5
    loop in which every offset is its own bucket.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, n, d = q.shape
    bo = np.asarray(bias_of_offset, dtype=np.float64)
    if bo.shape != (H, 2 * n - 1):
        raise ValueError("bias_of_offset must be [H, 2n - 1]")
    bias = np.ascontiguousarray(bo.T)                       # [2n - 1 "buckets", H]
    ident = np.ascontiguousarray(np.arange(2 * n - 1, dtype=np.int32))
    kvl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
    r, nrows = _rows_arg(rows, B, H, n)
    out = np.zeros((nrows, d), dtype=np.float64)
    rc = _load().oracle_t5bias_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(ident),
                                    int(bool(causal)), float(scale), _ptr(kvl), B, H, n, d,
                                    _ptr(r), nrows, _ptr(out),
                                    int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle thread start failed")
    return out if rows is not None else out.reshape(B, H, n, d)


def alibi_bias_of_offset(n: int, slopes) -> np.ndarray:
    """ALiBi as a bias per offset: b_h(delta) = -m_h * |delta| ("Relative position
    embeddings", section "Placement in the taxonomy"). Returns [H, 2n - 1], index
    delta + n - 1."""
    m = np.asarray(slopes, dtype=np.float64).reshape(-1)
    delta = np.arange(-(n - 1), n, dtype=np.float64)
    return -m[:, None] * np.abs(delta)[None, :]


def clipped_bias_of_offset(n: int, table, radius: int, heads: int) -> np.ndarray:
    """A learned scalar per offset, clipped at `radius` like the Shaw tables:
    b_h(delta) = table[h, clip(delta, radius) + radius]. table: [heads or 1, 2*radius + 1]
    (one row shared by every head). Returns [heads, 2n - 1], index delta + n - 1."""
    t = np.asarray(table, dtype=np.float64)
    if t.ndim != 2 or t.shape[1] != 2 * radius + 1 or t.shape[0] not in (1, heads):
        raise ValueError("table must be [heads or 1, 2*radius + 1]")
    out = np.empty((heads, 2 * n - 1), dtype=np.float64)
    for h in range(heads):
        row = t[h if t.shape[0] == heads else 0]
        for idx in range(2 * n - 1):
            out[h, idx] = row[clip(idx - (n - 1), radius) + radius]
    return out


def alibi_fwd(q, k, v, slopes, causal, scale, kv_len=None, rows=None, nthreads=None):
    """ALiBi attention forward, fp64: e_ij = scale * q_i . k_j - m_h |j - i|."""
    n = np.shape(q)[2]
    return offset_bias_fwd(q, k, v, alibi_bias_of_offset(n, slopes), causal, scale,
                           kv_len=kv_len, rows=rows, nthreads=nthreads)


def offset_table_fwd(q, k, v, table, radius, causal, scale, kv_len=None, rows=None,
                     nthreads=None):
    """Clipped per-offset scalar bias forward, fp64: e_ij = scale * q_i . k_j +
    table[h, clip(j - i, radius) + radius]."""
    H, n = np.shape(q)[1], np.shape(q)[2]
    return offset_bias_fwd(q, k, v, clipped_bias_of_offset(n, table, radius, H), causal, scale,
                           kv_len=kv_len, rows=rows, nthreads=nthreads)


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
