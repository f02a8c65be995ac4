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

Nothing here pins itself: tests/test_oracle_backward.py checks every gradient against
central finite differences of the C forward oracle, and the zero-table case against
PyTorch autograd of scaled dot-product attention.
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


def _offset_table_to_grid(table, n):
    """bucket_of_offset_table gives the bucket of offset j - i at index (j - i) + n - 1."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return table[(j - i) + n - 1]
