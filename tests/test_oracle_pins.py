"""Pins for the fp64 oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a number printed on the pages
(tests/golden/), a special case that reduces to a library routine, a closed form, an
invariant of the equations, or a brute-force restatement. They are chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle fails at
least one of them (tests/test_oracle_mutations.py plants such mistakes to check that).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, std=1.0):
    return rng.standard_normal(shape) * std


def _case(B, H, n, d, k, rng, table_std=0.3, with_aK=True, with_aV=True, Ht=None):
    Ht = H if Ht is None else Ht
    q, kk, v = (_rand((B, H, n, d), rng) for _ in range(3))
    aK = _rand((Ht, 2 * k + 1, d), rng, table_std) if with_aK else None
    aV = _rand((Ht, 2 * k + 1, d), rng, table_std) if with_aV else None
    return q, kk, v, aK, aV


def _sdpa(q, k, v, scale, causal=False, kv_len=None):
    """Library scaled dot-product attention in float64 on the CPU."""
    qt, kt, vt = (torch.from_numpy(np.asarray(x, dtype=np.float64)) for x in (q, k, v))
    B, H, n, d = qt.shape
    mask = torch.ones(B, 1, n, n, dtype=torch.bool)
    if kv_len is not None:
        for b in range(B):
            mask[b, :, :, int(kv_len[b]):] = False
    if causal:
        mask &= torch.ones(n, n, dtype=torch.bool).tril()
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                           scale=scale)
    return out.numpy()


# ---------------------------------------------------------------- printed values (I8)
def test_clip_examples_printed_on_the_page():
    g = json.load(open(os.path.join(GOLDEN, "clip_examples.json")))
    for ex in g["clip"]:
        assert oracle.clip(ex["x"], ex["k"]) == ex["clip"]
    # labels for k = 4 run -4..4 in table order w_{-k}..w_{k}
    lab = oracle.clip_labels(40, 40, 4)[20] - 4
    assert sorted(set(lab.tolist())) == g["labels_k4"]
    for lc in g["label_counts"]:
        n = 200
        labs = oracle.clip_labels(n, n, lc["k"])
        assert len(np.unique(labs)) == lc["count"] == 2 * lc["k"] + 1
        assert labs.min() == 0 and labs.max() == 2 * lc["k"]
    assert len(np.unique(oracle.clip_labels(50, 50, 0))) == g["k0_labels"]


def test_table_sizes_printed_on_the_page():
    g = json.load(open(os.path.join(GOLDEN, "clip_examples.json")))["param_counts"]
    rows = 2 * g["k"] + 1
    assert g["H"] * rows * g["d"] * 2 == g["per_head_both_tables"]
    assert rows * g["d"] * 2 == g["shared_both_tables"]


# --------------------------------------------------- hand-computed sign check (Q1)
def test_two_token_sign_and_table_order_by_hand():
    """n = 2, d = 1, k = 1, zero keys; only w^K_{+1} = c is non-zero.

    Row 0 sees key 1 at offset j - i = +1, so e_01 = scale*q_0*c and e_00 = 0; row 1 sees
    key 0 at offset -1 (w^K_{-1} = 0) so both logits are 0. With values v = (0, 1) and
    w^V_{+1} = 10 (other rows 0): z_0 = s*(1 + 10), z_1 = 1/2, with s = sigmoid(scale*c).
    Table row 0 is w_{-k}, so w_{+1} sits at row 2.
    """
    c, scale = 1.7, 0.5
    q = np.array([1.0, 1.0]).reshape(1, 1, 2, 1)
    k = np.zeros((1, 1, 2, 1))
    v = np.array([0.0, 1.0]).reshape(1, 1, 2, 1)
    aK = np.zeros((1, 3, 1)); aK[0, 2, 0] = c
    aV = np.zeros((1, 3, 1)); aV[0, 2, 0] = 10.0
    z = oracle.relattn_fwd(q, k, v, aK, aV, 1, False, scale)[0, 0, :, 0]
    s = 1.0 / (1.0 + math.exp(-scale * c))
    assert z[0] == pytest.approx(s * 11.0, rel=1e-14)
    assert z[1] == pytest.approx(0.5, rel=1e-14)


# ---------------------------------------------------- library reduction (I1)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("padded", [False, True])
def test_zero_tables_reduce_to_library_attention(causal, padded):
    rng = np.random.default_rng(1)
    B, H, n, d, k = 3, 2, 23, 16, 4
    q, kk, v, aK, aV = _case(B, H, n, d, k, rng)
    kv_len = np.array([23, 9, 1], dtype=np.int32) if padded else None
    scale = 1 / math.sqrt(d)
    z = oracle.relattn_fwd(q, kk, v, np.zeros_like(aK), np.zeros_like(aV), k, causal,
                           scale, kv_len=kv_len)
    ref = _sdpa(q, kk, v, scale, causal, kv_len)
    if padded and causal:
        # rows i >= 0 always keep j = 0 (kv_len >= 1), so no row is empty here
        pass
    np.testing.assert_allclose(z, ref, rtol=0, atol=1e-12)
    # tables absent (None) is the same thing
    z2 = oracle.relattn_fwd(q, kk, v, None, None, k, causal, scale, kv_len=kv_len)
    np.testing.assert_allclose(z2, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------- k = 0 closed forms (I2)
def test_k0_constant_key_table_leaves_alpha_and_constant_value_adds_exactly():
    rng = np.random.default_rng(2)
    B, H, n, d = 2, 3, 17, 8
    q, kk, v, _, _ = _case(B, H, n, d, 0, rng)
    wK = _rand((H, 1, d), rng, 1.0)
    wV = _rand((H, 1, d), rng, 1.0)
    scale = 0.37
    base = _sdpa(q, kk, v, scale)
    # k = 0: every pair uses w_0; q_i . w_0 is constant along the row -> alpha unchanged
    z_k = oracle.relattn_fwd(q, kk, v, wK, None, 0, False, scale)
    np.testing.assert_allclose(z_k, base, rtol=0, atol=1e-12)
    # constant value edge: sum_j alpha_ij = 1, so z_i gains exactly w^V_0
    z_kv = oracle.relattn_fwd(q, kk, v, wK, wV, 0, False, scale)
    np.testing.assert_allclose(z_kv, base + wV[None, :, :, :].transpose(0, 1, 2, 3)
                               .reshape(1, H, 1, d), rtol=0, atol=1e-12)


# ------------------------------------------------------------- causal row 0 (I3)
def test_causal_first_row_is_value_plus_offset_zero_edge():
    rng = np.random.default_rng(3)
    B, H, n, d, k = 2, 2, 9, 4, 3
    q, kk, v, aK, aV = _case(B, H, n, d, k, rng)
    z = oracle.relattn_fwd(q, kk, v, aK, aV, k, True, 0.5)
    # one allowed key (j = 0), offset 0 -> table row k
    np.testing.assert_allclose(z[:, :, 0, :], v[:, :, 0, :] + aV[None, :, k, :],
                               rtol=0, atol=1e-14)


# ------------------------------------------------------- shift invariance (I4)
@pytest.mark.parametrize("causal", [False, True])
def test_relative_only_dependence_under_a_shift(causal):
    """Put m tokens at offset s in a longer buffer; filler keys are made unreachable by a
    huge negative logit (exp underflows to exactly 0 in fp64). Outputs at s..s+m-1 must
    equal the unshifted outputs (translation equivariance of clip(j - i))."""
    rng = np.random.default_rng(4)
    H, m, d, k, s, n = 2, 11, 6, 3, 7, 25
    q, kk, v, aK, aV = _case(1, H, m, d, k, rng)
    # extra channel: queries carry 1, real keys 0, fillers -1e6 -> filler logit -1e6*scale
    ext = lambda x, val: np.concatenate([x, np.full(x.shape[:-1] + (1,), val)], axis=-1)
    qe = ext(q, 1.0)
    ke = ext(kk, 0.0)
    ve = ext(v, 0.0)
    aKe = ext(aK, 0.0)
    aVe = ext(aV, 0.0)
    Q = np.zeros((1, H, n, d + 1)); K = np.zeros_like(Q); V = np.zeros_like(Q)
    K[..., d] = -1e6
    Q[:, :, s:s + m] = qe; K[:, :, s:s + m] = ke; V[:, :, s:s + m] = ve
    ref = oracle.relattn_fwd(qe, ke, ve, aKe, aVe, k, causal, 0.25)
    big = oracle.relattn_fwd(Q, K, V, aKe, aVe, k, causal, 0.25)
    np.testing.assert_allclose(big[:, :, s:s + m], ref, rtol=0, atol=1e-12)


# ------------------------------------------------ brute force / split form (I5, I6)
@pytest.mark.parametrize("n,k", [(1, 0), (7, 0), (9, 1), (13, 2), (16, 15), (16, 19),
                                 (33, 4), (40, 39)])
@pytest.mark.parametrize("causal", [False, True])
def test_materialised_split_and_loop_agree(n, k, causal):
    rng = np.random.default_rng(100 + n * 7 + k)
    B, H, d = 2, 2, 5
    q, kk, v, aK, aV = _case(B, H, n, d, k, rng)
    kv_len = np.array([n, max(1, n // 2)], dtype=np.int32)
    scale = 0.4
    z_loop = oracle.relattn_fwd(q, kk, v, aK, aV, k, causal, scale, kv_len=kv_len)
    z_mat = brute.materialised(q, kk, v, aK, aV, k, causal, scale, kv_len=kv_len)
    z_split, beta = brute.split(q, kk, v, aK, aV, k, causal, scale, kv_len=kv_len)
    np.testing.assert_allclose(z_loop, z_mat, rtol=0, atol=1e-12)
    np.testing.assert_allclose(z_split, z_mat, rtol=0, atol=1e-12)
    # bins of a probability row sum to one
    np.testing.assert_allclose(beta.sum(-1), 1.0, rtol=0, atol=1e-12)
    if k >= n - 1:
        # no clipping: each bin holds at most one key, so beta is alpha re-indexed by j - i
        nz = (beta > 0).sum(-1)
        assert (nz <= np.minimum(n, 2 * k + 1)).all()
        for i in range(n):
            for j in range(n):
                r = j - i + k
                if causal and j > i:
                    continue
                if j >= kv_len[0]:
                    continue
                assert beta[0, 0, i, r] > 0


def test_shared_tables_equal_broadcast_per_head_tables():
    rng = np.random.default_rng(5)
    B, H, n, d, k = 2, 3, 12, 4, 2
    q, kk, v, aK, aV = _case(B, H, n, d, k, rng, Ht=1)
    z_shared = oracle.relattn_fwd(q, kk, v, aK, aV, k, False, 0.5, table_head_stride=0)
    z_per = oracle.relattn_fwd(q, kk, v, np.repeat(aK, H, 0), np.repeat(aV, H, 0), k, False,
                               0.5)
    np.testing.assert_allclose(z_shared, z_per, rtol=0, atol=0)


def test_sampled_rows_match_full_output():
    rng = np.random.default_rng(6)
    B, H, n, d, k = 2, 2, 19, 3, 2
    q, kk, v, aK, aV = _case(B, H, n, d, k, rng)
    full = oracle.relattn_fwd(q, kk, v, aK, aV, k, True, 0.3)
    rows = np.array([0, 5, 18, 19, 40, B * H * n - 1])
    part = oracle.relattn_fwd(q, kk, v, aK, aV, k, True, 0.3, rows=rows)
    np.testing.assert_array_equal(part, full.reshape(-1, d)[rows])


def test_empty_row_is_zero():
    rng = np.random.default_rng(7)
    q, kk, v, aK, aV = _case(2, 1, 5, 3, 1, rng)
    z = oracle.relattn_fwd(q, kk, v, aK, aV, 1, False, 1.0,
                           kv_len=np.array([0, 5], dtype=np.int32))
    assert (z[0] == 0).all()
    assert np.abs(z[1]).sum() > 0


# ------------------------------------------------------- key-only / T5 (I7, I9)
def test_key_only_equals_zero_value_table():
    rng = np.random.default_rng(8)
    q, kk, v, aK, aV = _case(2, 2, 14, 6, 3, rng)
    a = oracle.relattn_fwd(q, kk, v, aK, None, 3, True, 0.5)
    b = oracle.relattn_fwd(q, kk, v, aK, np.zeros_like(aV), 3, True, 0.5)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_t5_constant_bias_per_head_reduces_to_library_attention(causal):
    rng = np.random.default_rng(9)
    B, H, n, d = 2, 3, 40, 8
    q, kk, v, _, _ = _case(B, H, n, d, 0, rng)
    bias = np.tile(rng.standard_normal((1, H)) * 3, (32, 1))   # same value in every bucket
    z = oracle.t5bias_fwd(q, kk, v, bias, 32, 128, True, causal, 1.0)
    np.testing.assert_allclose(z, _sdpa(q, kk, v, 1.0, causal), rtol=0, atol=1e-12)


def test_t5_bias_equals_shaw_style_materialised_bias():
    """T5 logit = scale*q.k + b[bucket(j-i), h]: compare with an explicit n x n bias."""
    rng = np.random.default_rng(10)
    B, H, n, d = 1, 2, 30, 4
    q, kk, v, _, _ = _case(B, H, n, d, 0, rng)
    bias = rng.standard_normal((32, H))
    lab = oracle.t5_labels(n, n, 32, 20, True)
    z = oracle.t5bias_fwd(q, kk, v, bias, 32, 20, True, False, 0.7)
    for h in range(H):
        e = 0.7 * q[0, h] @ kk[0, h].T + bias[lab, h]
        p = np.exp(e - e.max(1, keepdims=True))
        ref = (p / p.sum(1, keepdims=True)) @ v[0, h]
        np.testing.assert_allclose(z[0, h], ref, rtol=0, atol=1e-12)
