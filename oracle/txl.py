"""fp64 Transformer-XL relative attention (the four-term score), for tests.

TEST INFRASTRUCTURE ONLY (same rule as the rest of oracle/).

Source: "Relative Position Encoding in Transformer-XL" page (the four-term score and the
roles of u and v) and "Relative position embeddings" page, section "Transformer-XL":

    A_ij = q_i . k_j            (a) content-content
         + q_i . r_ij           (b) content-position
         + u . k_j              (c) global content bias
         + v . r_ij             (d) global position bias
    alpha_i = softmax_j(scale * A_ij) over the allowed keys,   z_i = sum_j alpha_ij v_j

with r_ij = W_{k,R} r(i, j), the projected encoding of the pair's relative offset: the
caller passes these projected vectors as a table `rel` [H, 2n - 1, d] indexed by the offset
j - i + n - 1 (the pages write the subscript i - j in the formula and describe negative
distances as keys before the query in the prose; a table over all offsets holds either
convention, and this one uses j - i like the rest of the library). `scale` multiplies the
whole score (the pages print the score without it; 1/sqrt(d) is the usual choice).
u and v are per head here ([H, d]); the value projection's input v_j is named `val` below
to keep it apart from the bias vector v, which is `vb`.

Each term is formed on its own and the four are summed, as the formula is written; the
offset gather of (b) and (d) is plain indexing of the full product with the table (the
"shift" the pages mention is this reindexing).
"""
from __future__ import annotations

import numpy as np


def txl_fwd(q, k, val, rel, u, vb, causal, scale, kv_len=None):
    """q, k, val: [B, H, n, d]; rel: [H, 2n - 1, d]; u, vb: [H, d]. Returns z [B, H, n, d]."""
    q, k, val = (np.asarray(x, dtype=np.float64) for x in (q, k, val))
    rel = np.asarray(rel, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    vb = np.asarray(vb, dtype=np.float64)
    B, H, n, d = q.shape
    if rel.shape != (H, 2 * n - 1, d) or u.shape != (H, d) or vb.shape != (H, d):
        raise ValueError("rel must be [H, 2n - 1, d], u and vb [H, d]")
    i_idx = np.arange(n)[:, None]
    j_idx = np.arange(n)[None, :]
    off = (j_idx - i_idx) + (n - 1)                       # table row of every (i, j)
    out = np.zeros_like(q)
    for b in range(B):
        valid = n if kv_len is None else max(0, min(int(kv_len[b]), n))
        ok = np.broadcast_to(j_idx < valid, (n, n))
        if causal:
            ok = ok & (j_idx <= i_idx)
        for h in range(H):
            term_a = q[b, h] @ k[b, h].T                          # [n, n]
            term_b = (q[b, h] @ rel[h].T)[i_idx, off]             # q_i . r_ij
            term_c = np.broadcast_to(k[b, h] @ u[h], (n, n))      # u . k_j, same for every i
            term_d = (rel[h] @ vb[h])[off]                        # v . r_ij
            e = scale * (term_a + term_b + term_c + term_d)
            e = np.where(ok, e, -np.inf)
            m = e.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            p = np.where(ok, np.exp(e - m), 0.0)
            l = p.sum(axis=1, keepdims=True)
            alpha = np.where(l > 0, p / np.where(l > 0, l, 1.0), 0.0)
            out[b, h] = alpha @ val[b, h]
    return out


def sinusoid_table(n, d_model):
    """The sinusoidal encodings of every relative offset of a length-n sequence, the r of the
    Transformer-XL score before its projection W_{k,R}: row o holds offset o - (n - 1), and
    for an offset p the components are PE(p, 2i) = sin(p / 10000^(2i / d_model)) and
    PE(p, 2i + 1) = cos(p / 10000^(2i / d_model)) ("Self-Attention with Relative Position
    Representations" page, the original Transformer's position encodings; "Relative Position
    Encoding in Transformer-XL" page: r is this fixed sinusoid of the distance). fp64,
    [2n - 1, d_model]; d_model even."""
    if d_model % 2:
        raise ValueError("d_model must be even")
    pos = np.arange(-(n - 1), n, dtype=np.float64)[:, None]          # offsets
    i2 = np.arange(0, d_model, 2, dtype=np.float64)[None, :]          # 2i
    ang = pos / np.power(10000.0, i2 / d_model)
    out = np.empty((2 * n - 1, d_model), dtype=np.float64)
    out[:, 0::2] = np.sin(ang)
    out[:, 1::2] = np.cos(ang)
    return out
