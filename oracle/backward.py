"""fp64 gradients of relation-aware attention and of the T5 bucketed-bias attention.

TEST INFRASTRUCTURE ONLY (same rule as the rest of oracle/).

The pages state only the forward pass (Shaw et al., eq. 3, eq. 4 and the softmax; T5 as
summarised under "Relative position embeddings"). The gradients below are the plain chain
rule through those definitions, written per (b, h) with numpy:

  e_ij  = scale * q_i . (k_j + a^K_ij)             (Shaw)   or  scale * q_i . k_j + b(j - i)  (T5)
  p_ij  = softmax_j(e_ij) over the allowed keys j
  z_i   = sum_j p_ij (v_j + a^V_ij)                (a^V term absent: v_j only)

  dp_ij = dz_i . (v_j + a^V_ij)
  de_ij = p_ij (dp_ij - sum_j' p_ij' dp_ij')       (softmax Jacobian)
  dq_i  = scale * sum_j de_ij (k_j + a^K_ij)
  dk_j  = scale * sum_i de_ij q_i
  dv_j  = sum_i p_ij dz_i
  dw^K_r = scale * sum_{(i,j): r_ij = r} de_ij q_i,   dw^V_r = sum_{(i,j): r_ij = r} p_ij dz_i
  dbias[bucket, h] = sum_{(b,i,j): bucket(j - i) = bucket} de_ij

with r_ij = clip(j - i, k) + k. The sums over (i, j) with one label are taken through the
bins gamma_ir = sum_{j: r_ij = r} de_ij and beta_ir = sum_{j: r_ij = r} p_ij, so the n x n x d
edge tensors are never built. A row with no allowed key has p = 0 and contributes nothing.

The same chain rule gives the gradients of the labelled-edge forward (r_ij from a label
matrix), of the clipped per-offset scalar table (dtable[h, r] = sum of de_ij over the pairs
with clip(j - i, R) + R = r) and of ALiBi with respect to its slopes (d e_ij / d m_h =
-|j - i|).

Nothing here pins itself: tests/test_oracle_backward.py checks every gradient against
central finite differences of the forward oracle (the C loop), the zero-table case against
PyTorch autograd of scaled dot-product attention, and the labelled form with clip labels
against the Shaw gradients.
"""
from __future__ import annotations

import numpy as np

from . import t5 as _t5


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def _mask(n, causal, valid):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    ok = np.broadcast_to(j < valid, (n, n))
    if causal:
        ok = ok & (j <= i)
    return ok


def _softmax_rows(e, ok):
    e = np.where(ok, e, -np.inf)
    m = e.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.where(ok, np.exp(e - m), 0.0)
    l = p.sum(axis=1, keepdims=True)
    return np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)


def _bins(x, lab, nbins):
    """out[i, r] = sum over j with lab[i, j] = r of x[i, j]."""
    out = np.zeros((x.shape[0], nbins), dtype=np.float64)
    rows = np.repeat(np.arange(x.shape[0]), x.shape[1])
    np.add.at(out, (rows, lab.reshape(-1)), x.reshape(-1))
    return out


def relattn_bwd(q, k, v, aK, aV, dz, clip_k, causal, scale, kv_len=None,
                table_head_stride=None):
    """Gradients (dq, dk, dv, daK, daV) of the Shaw forward, fp64.

    q, k, v, dz: [B, H, n, d]. aK / aV: [H_t, 2*clip_k + 1, d] or None (term absent; its
    gradient is then None). table_head_stride: elements between heads' tables (default
    (2k+1)*d; 0 = one table shared by all heads, whose gradient sums over the heads).
    """
    q, k, v, dz = (_f64(x) for x in (q, k, v, dz))
    B, H, n, d = q.shape
    W = 2 * clip_k + 1
    ths = W * d if table_head_stride is None else int(table_head_stride)
    aKf = None if aK is None else _f64(aK).reshape(-1)
    aVf = None if aV is None else _f64(aV).reshape(-1)
    daK = None if aK is None else np.zeros_like(aKf)
    daV = None if aV is None else np.zeros_like(aVf)
    i_idx = np.arange(n)[:, None]
    j_idx = np.arange(n)[None, :]
    lab = np.clip(j_idx - i_idx, -clip_k, clip_k) + clip_k          # [n, n]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        valid = n if kv_len is None else max(0, min(int(kv_len[b]), n))
        ok = _mask(n, causal, valid)
        for h in range(H):
            qh, kh, vh, gz = q[b, h], k[b, h], v[b, h], dz[b, h]
            wK = None if aKf is None else aKf[h * ths: h * ths + W * d].reshape(W, d)
            wV = None if aVf is None else aVf[h * ths: h * ths + W * d].reshape(W, d)
            e = qh @ kh.T
            if wK is not None:
                e = e + (qh @ wK.T)[i_idx, lab]
            p = _softmax_rows(scale * e, ok)
            dp = gz @ vh.T
            if wV is not None:
                dp = dp + (gz @ wV.T)[i_idx, lab]
            de = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (de @ kh)
            dk[b, h] = scale * (de.T @ qh)
            dv[b, h] = p.T @ gz
            if wK is not None:
                gamma = _bins(de, lab, W)
                dq[b, h] += scale * (gamma @ wK)
                daK[h * ths: h * ths + W * d] += (scale * (gamma.T @ qh)).reshape(-1)
            if wV is not None:
                beta = _bins(p, lab, W)
                daV[h * ths: h * ths + W * d] += (beta.T @ gz).reshape(-1)
    if daK is not None:
        daK = daK.reshape(np.shape(aK))
    if daV is not None:
        daV = daV.reshape(np.shape(aV))
    return dq, dk, dv, daK, daV


def t5bias_bwd(q, k, v, bias, dz, num_buckets, max_distance, bidirectional, causal, scale,
               kv_len=None):
    """Gradients (dq, dk, dv, dbias) of the T5 bucketed-bias forward, fp64.

    bias: [num_buckets, H] (shared by the batch, so its gradient sums over it).
    """
    q, k, v, dz, bias = (_f64(x) for x in (q, k, v, dz, bias))
    B, H, n, d = q.shape
    lab = _offset_table_to_grid(np.asarray(
        _t5.bucket_of_offset_table(n, num_buckets, max_distance, bool(bidirectional)),
        dtype=np.int64), n)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dbias = np.zeros_like(bias)
    for b in range(B):
        valid = n if kv_len is None else max(0, min(int(kv_len[b]), n))
        ok = _mask(n, causal, valid)
        for h in range(H):
            qh, kh, vh, gz = q[b, h], k[b, h], v[b, h], dz[b, h]
            e = scale * (qh @ kh.T) + bias[lab, h]
            p = _softmax_rows(e, ok)
            dp = gz @ vh.T
            de = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (de @ kh)
            dk[b, h] = scale * (de.T @ qh)
            dv[b, h] = p.T @ gz
            np.add.at(dbias[:, h], lab.reshape(-1), de.reshape(-1))
    return dq, dk, dv, dbias


def labeled_bwd(q, k, v, aK, aV, dz, labels, causal, scale, kv_len=None,
                table_head_stride=None):
    """Gradients (dq, dk, dv, daK, daV) of the labelled-edge forward (oracle.labeled_fwd),
    fp64: the chain rule above with r_ij = L_b[i, j] in place of clip(j - i, k) + k.

    labels: [n, n] or [B, n, n] integer labels; aK / aV: [H_t, num_labels, d] or None.
    """
    q, k, v, dz = (_f64(x) for x in (q, k, v, dz))
    B, H, n, d = q.shape
    ref = aK if aK is not None else aV
    W = 0 if ref is None else np.shape(ref)[1]
    ths = W * d if table_head_stride is None else int(table_head_stride)
    aKf = None if aK is None else _f64(aK).reshape(-1)
    aVf = None if aV is None else _f64(aV).reshape(-1)
    daK = None if aK is None else np.zeros_like(aKf)
    daV = None if aV is None else np.zeros_like(aVf)
    L = np.asarray(labels, dtype=np.int64)
    i_idx = np.arange(n)[:, None]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        lab = L if L.ndim == 2 else L[b]
        valid = n if kv_len is None else max(0, min(int(kv_len[b]), n))
        ok = _mask(n, causal, valid)
        for h in range(H):
            qh, kh, vh, gz = q[b, h], k[b, h], v[b, h], dz[b, h]
            wK = None if aKf is None else aKf[h * ths: h * ths + W * d].reshape(W, d)
            wV = None if aVf is None else aVf[h * ths: h * ths + W * d].reshape(W, d)
            e = qh @ kh.T
            if wK is not None:
                e = e + (qh @ wK.T)[i_idx, lab]
            p = _softmax_rows(scale * e, ok)
            dp = gz @ vh.T
            if wV is not None:
                dp = dp + (gz @ wV.T)[i_idx, lab]
            de = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (de @ kh)
            dk[b, h] = scale * (de.T @ qh)
            dv[b, h] = p.T @ gz
            if wK is not None:
                gamma = _bins(de, lab, W)
                dq[b, h] += scale * (gamma @ wK)
                daK[h * ths: h * ths + W * d] += (scale * (gamma.T @ qh)).reshape(-1)
            if wV is not None:
                beta = _bins(p, lab, W)
                daV[h * ths: h * ths + W * d] += (beta.T @ gz).reshape(-1)
    if daK is not None:
        daK = daK.reshape(np.shape(aK))
    if daV is not None:
        daV = daV.reshape(np.shape(aV))
    return dq, dk, dv, daK, daV


def offset_table_bwd(q, k, v, table, radius, dz, causal, scale, kv_len=None):
    """Gradients (dq, dk, dv, dtable) of the clipped per-offset scalar bias forward
    (oracle.offset_table_fwd): e_ij = scale q_i.k_j + table[h, clip(j - i, R) + R], so
    dtable[h, r] = sum over (b, i, j) with clip(j - i, R) + R = r of de_ij. table: [H or 1,
    2R + 1] (one shared row sums over the heads)."""
    q, k, v, dz = (_f64(x) for x in (q, k, v, dz))
    t = _f64(table)
    B, H, n, d = q.shape
    R = int(radius)
    i_idx = np.arange(n)[:, None]
    j_idx = np.arange(n)[None, :]
    lab = np.clip(j_idx - i_idx, -R, R) + R
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dt = np.zeros_like(t)
    for b in range(B):
        valid = n if kv_len is None else max(0, min(int(kv_len[b]), n))
        ok = _mask(n, causal, valid)
        for h in range(H):
            row = h if t.shape[0] == H else 0
            qh, kh, vh, gz = q[b, h], k[b, h], v[b, h], dz[b, h]
            p = _softmax_rows(scale * (qh @ kh.T) + t[row][lab], ok)
            dp = gz @ vh.T
            de = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (de @ kh)
            dk[b, h] = scale * (de.T @ qh)
            dv[b, h] = p.T @ gz
            np.add.at(dt[row], lab.reshape(-1), de.reshape(-1))
    return dq, dk, dv, dt


def alibi_slope_bwd(q, k, v, slopes, dz, causal, scale, kv_len=None):
    """Gradient of the ALiBi forward with respect to its slopes (fixed in the method, but
    the derivative is d e_ij / d m_h = -|j - i|): dm[h] = -sum over (b, i, j) of |j - i| de_ij.
    Returns (dq, dk, dv, dslopes)."""
    q, k, v, dz = (_f64(x) for x in (q, k, v, dz))
    m = _f64(slopes).reshape(-1)
    B, H, n, d = q.shape
    dist = np.abs(np.arange(n)[None, :] - np.arange(n)[:, None]).astype(np.float64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dm = np.zeros_like(m)
    for b in range(B):
        valid = n if kv_len is None else max(0, min(int(kv_len[b]), n))
        ok = _mask(n, causal, valid)
        for h in range(H):
            qh, kh, vh, gz = q[b, h], k[b, h], v[b, h], dz[b, h]
            p = _softmax_rows(scale * (qh @ kh.T) - m[h] * dist, ok)
            dp = gz @ vh.T
            de = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (de @ kh)
            dk[b, h] = scale * (de.T @ qh)
            dv[b, h] = p.T @ gz
            dm[h] -= float((de * dist).sum())
    return dq, dk, dv, dm


def _offset_table_to_grid(table, n):
    """bucket_of_offset_table gives the bucket of offset j - i at index (j - i) + n - 1."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return table[(j - i) + n - 1]
