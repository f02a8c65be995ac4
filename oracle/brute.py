"""Two more numpy fp64 statements of Shaw relation-aware attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY (same rule as the rest of oracle/).

materialised(): the naive form the "Self-Attention with Relative Position Representations" page calls prohibitive ("Efficient
Implementation: How the Method Scales", opening paragraph): build the n x n x d edge
tensors a^K_ij = w^K[clip(j-i,k)+k] and a^V_ij = w^V[clip(j-i,k)+k] explicitly, add them
to the keys and values, and apply eq. 4, the softmax and eq. 3 as written.

split(): the rewrite the same section describes, eq. 5 for the logits
    e_ij = scale * (q_i . k_j + q_i . a^K_ij),
where the second term is gathered from the small product R = Q . W^K^T
(R[i, r] = q_i . w^K_r, r = clip(j-i,k)+k), and the two-sum split of eq. 3,
    z_i = sum_j alpha_ij v_j + sum_j alpha_ij a^V_ij.
The second sum only sees 2k+1 distinct rows of W^V, so it equals beta_i . W^V with the
bins beta_ir = sum over {j : clip(j-i,k)+k = r} of alpha_ij. (That binning is the plain
algebraic reading of "the same approach can be used" for eq. 3; the pages do not spell
it out.) Returning beta lets tests check sum_r beta_ir = 1.
"""
from __future__ import annotations

import numpy as np


def _allowed(n, i_idx, j_idx, causal, valid):
    ok = j_idx[None, :] < valid
    if causal:
        ok = ok & (j_idx[None, :] <= i_idx[:, None])
    return np.broadcast_to(ok, (len(i_idx), len(j_idx)))


def _labels(n, clip_k):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return np.clip(j - i, -clip_k, clip_k) + clip_k


def _tables(tab, h, ths, rows, d):
    if tab is None:
        return None
    flat = np.asarray(tab, dtype=np.float64).reshape(-1)
    return flat[h * ths: h * ths + rows * d].reshape(rows, d)


def _softmax_rows(e, ok):
    e = np.where(ok, e, -np.inf)
    m = e.max(axis=1, keepdims=True)
    has = np.isfinite(m)
    m = np.where(has, m, 0.0)
    p = np.where(ok, np.exp(e - m), 0.0)
    l = p.sum(axis=1, keepdims=True)
    return np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)


def materialised(q, k, v, aK, aV, clip_k, causal, scale, kv_len=None, table_head_stride=None,
                 labels=None, num_labels=None):
    """labels: optional edge labels ([n, n] or [B, n, n]) in place of clip(j - i, k) + k, for
    tables of num_labels rows (the general labelled graph of the "Self-Attention with Relative Position Representations" page, section
    "Relation-Aware Self-Attention: The Core Modification")."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, n, d = q.shape
    rows = 2 * clip_k + 1 if labels is None else int(num_labels)
    ths = rows * d if table_head_stride is None else table_head_stride
    out = np.zeros_like(q)
    idx = np.arange(n)
    for b in range(B):
        if labels is None:
            lab = _labels(n, clip_k)
        else:
            L = np.asarray(labels, dtype=np.int64)
            lab = L if L.ndim == 2 else L[b]
        valid = n if kv_len is None else min(int(kv_len[b]), n)
        ok = _allowed(n, idx, idx, causal, valid)
        for h in range(H):
            wK = _tables(aK, h, ths, rows, d)
            wV = _tables(aV, h, ths, rows, d)
            AK = wK[lab] if wK is not None else np.zeros((n, n, d))   # [i, j, d]
            AV = wV[lab] if wV is not None else np.zeros((n, n, d))
            keys = k[b, h][None, :, :] + AK                            # k_j + a^K_ij
            e = scale * np.einsum("ic,ijc->ij", q[b, h], keys)
            alpha = _softmax_rows(e, ok)
            vals = v[b, h][None, :, :] + AV                            # v_j + a^V_ij
            out[b, h] = np.einsum("ij,ijc->ic", alpha, vals)
    return out


def split(q, k, v, aK, aV, clip_k, causal, scale, kv_len=None, table_head_stride=None):
    """Returns (z, beta) with beta[b, h, i, r] the value bins."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, n, d = q.shape
    W = 2 * clip_k + 1
    ths = W * d if table_head_stride is None else table_head_stride
    lab = _labels(n, clip_k)
    out = np.zeros_like(q)
    beta = np.zeros((B, H, n, W))
    idx = np.arange(n)
    for b in range(B):
        valid = n if kv_len is None else min(int(kv_len[b]), n)
        ok = _allowed(n, idx, idx, causal, valid)
        for h in range(H):
            wK = _tables(aK, h, ths, W, d)
            wV = _tables(aV, h, ths, W, d)
            content = q[b, h] @ k[b, h].T                              # term 1 of eq. 5
            if wK is not None:
                R = q[b, h] @ wK.T                                     # [n, 2k+1]
                rel = np.take_along_axis(R, lab, axis=1)               # term 2 of eq. 5
            else:
                rel = 0.0
            alpha = _softmax_rows(scale * (content + rel), ok)
            z = alpha @ v[b, h]
            for r in range(W):
                beta[b, h, :, r] = np.where(lab == r, alpha, 0.0).sum(axis=1)
            if wV is not None:
                z = z + beta[b, h] @ wV
            out[b, h] = z
    return out, beta
