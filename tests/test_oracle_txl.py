"""Pins for the Transformer-XL oracle (oracle/txl.py).

The pages give the four-term score and no numbers. What fixes the expected values:
  * zero encodings and biases: PyTorch scaled dot-product attention (library routine);
  * u = v: the score is (q_i + u) . (k_j + r_ij), the Shaw form with an unclipped table,
    so the C loop of the Shaw oracle (pinned on its own) must agree;
  * zero queries and keys: only term (d) is left, a scalar per offset, which the offset-bias
    oracle (pinned on its own) computes;
  * zero queries and encodings: only term (c) is left, u . k_j for every row: library
    attention with u as every row's query.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import txl


def _setup(B, H, n, d, seed):
    rng = np.random.default_rng(seed)
    q, k, val = (rng.standard_normal((B, H, n, d)) for _ in range(3))
    rel = rng.standard_normal((H, 2 * n - 1, d)) * 0.5
    u = rng.standard_normal((H, d))
    vb = rng.standard_normal((H, d))
    return q, k, val, rel, u, vb


@pytest.mark.parametrize("causal", [False, True])
def test_zero_encodings_and_biases_is_library_attention(causal):
    q, k, val, rel, u, vb = _setup(2, 3, 10, 4, 0)
    z = txl.txl_fwd(q, k, val, np.zeros_like(rel), np.zeros_like(u), np.zeros_like(vb),
                    causal, 0.5)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(val), is_causal=causal,
        scale=0.5).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal,kvl", [(False, None), (True, None), (False, [6, 11])])
def test_equal_biases_is_shaw_with_an_unclipped_table(causal, kvl):
    B, H, n, d = 2, 2, 11, 3
    q, k, val, rel, u, _ = _setup(B, H, n, d, 1)
    z = txl.txl_fwd(q, k, val, rel, u, u, causal, 0.7, kv_len=kvl)
    # (q + u) . (k_j + r_ij): the Shaw score with clip k = n - 1, whose row (j - i) + n - 1
    # is the table row of the pair
    shaw = oracle.relattn_fwd(q + u[None, :, None, :], k, val, rel, None, n - 1, causal, 0.7,
                              kv_len=kvl)
    np.testing.assert_allclose(z, shaw, rtol=1e-12, atol=1e-12)


def test_global_position_bias_alone_is_a_scalar_per_offset():
    B, H, n, d = 1, 2, 9, 4
    _, _, val, rel, u, vb = _setup(B, H, n, d, 2)
    zero = np.zeros((B, H, n, d))
    z = txl.txl_fwd(zero, zero, val, rel, u, vb, False, 0.8)
    bias = 0.8 * np.einsum("hod,hd->ho", rel, vb)        # scale * v . r for every offset
    ref = oracle.offset_bias_fwd(zero, zero, val, bias, False, 1.0)
    np.testing.assert_allclose(z, ref, rtol=1e-12, atol=1e-12)


def test_global_content_bias_alone_is_attention_with_u_as_query():
    B, H, n, d = 2, 2, 8, 5
    _, k, val, rel, u, vb = _setup(B, H, n, d, 3)
    zero = np.zeros((B, H, n, d))
    z = txl.txl_fwd(zero, k, val, np.zeros_like(rel), u, vb, True, 0.6)
    uq = np.broadcast_to(u[None, :, None, :], (B, H, n, d)).copy()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(uq), torch.from_numpy(k), torch.from_numpy(val), is_causal=True,
        scale=0.6).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-12, atol=1e-12)


def test_sinusoid_table_dot_products_depend_only_on_the_offset_difference():
    """sin(a) sin(b) + cos(a) cos(b) = cos(a - b): the dot product of the encodings of two
    offsets is sum_i cos((p - p') w_i), a function of p - p' alone. Checked on every pair of
    rows against the one-dimensional cosine sum, so a wrong frequency, a swapped sin/cos or a
    shifted offset row fails."""
    n, dm = 17, 12
    r = txl.sinusoid_table(n, dm)
    assert r.shape == (2 * n - 1, dm)
    w = 1.0 / np.power(10000.0, np.arange(0, dm, 2) / dm)
    offs = np.arange(-(n - 1), n)
    gram = r @ r.T
    diff = offs[:, None] - offs[None, :]
    expect = np.cos(diff[:, :, None] * w[None, None, :]).sum(axis=2)
    np.testing.assert_allclose(gram, expect, rtol=0, atol=1e-12)


def test_sinusoid_table_offset_zero_and_sign():
    """Offset 0 (row n - 1) is [0, 1, 0, 1, ...]; the sine components are odd in the offset and
    the cosine components even, and the row of offset +1 has a positive first component."""
    n, dm = 9, 8
    r = txl.sinusoid_table(n, dm)
    np.testing.assert_array_equal(r[n - 1], np.tile([0.0, 1.0], dm // 2))
    np.testing.assert_allclose(r[n - 1 + 3, 0::2], -r[n - 1 - 3, 0::2], atol=1e-15)
    np.testing.assert_allclose(r[n - 1 + 3, 1::2], r[n - 1 - 3, 1::2], atol=1e-15)
    assert r[n, 0] > 0.0
