"""Pins for the scalar offset-bias oracle (ALiBi and the clipped per-offset table).

The pages state the form of these biases ("Relative position embeddings" page, sections
"T5" and "Placement in the taxonomy": a scalar per head added to the logit, which for
ALiBi is -m_h |j - i|) and print no numbers for them. What fixes the expected values:
  * zero bias: PyTorch scaled dot-product attention in float64 (library routine);
  * any bias per offset: the same library routine with the bias grid as an additive mask;
  * the page's own statement that ALiBi is the T5 bias with a linear table: the T5 path
    of the oracle (its own bucketing code) with bias[bucket] = -m * |offset of bucket|,
    at lengths where every offset has its own bucket;
  * closed forms: with zero queries the weights are exp(-m|j - i|) normalised, read off
    one-hot values; a 2-token sign check of the clipped table by hand;
  * the softmax's shift invariance (a constant added to every offset changes nothing).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _sdpa(q, k, v, grid, causal, scale, kv_len=None):
    """float64 library attention with an additive float mask [H, n, n] (or None)."""
    B, H, n, d = q.shape
    mask = np.zeros((B, H, n, n))
    if grid is not None:
        mask += grid[None]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    for b in range(B):
        ok = np.ones((n, n), dtype=bool)
        if kv_len is not None:
            ok &= j < kv_len[b]
        if causal:
            ok &= j <= i
        mask[b, :, ~ok] = -np.inf
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask), scale=scale)
    return out.numpy()


def _grid(bias_of_offset, n):
    """[H, n, n] grid with grid[h, i, j] = bias_of_offset[h, (j - i) + n - 1], by loops."""
    H = bias_of_offset.shape[0]
    g = np.empty((H, n, n))
    for h in range(H):
        for i in range(n):
            for j in range(n):
                g[h, i, j] = bias_of_offset[h, (j - i) + n - 1]
    return g


def _inputs(B, H, n, d, seed):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((B, H, n, d)) for _ in range(3))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_slopes_is_library_attention(causal):
    q, k, v = _inputs(2, 3, 11, 4, 0)
    got = oracle.alibi_fwd(q, k, v, np.zeros(3), causal, 0.5)
    ref = _sdpa(q, k, v, None, causal, 0.5)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal,kvl", [(False, None), (True, None), (False, [3, 9])])
def test_any_offset_bias_is_library_attention_with_mask(causal, kvl):
    B, H, n, d = 2, 2, 9, 3
    q, k, v = _inputs(B, H, n, d, 1)
    bo = np.random.default_rng(2).standard_normal((H, 2 * n - 1)) * 2.0
    got = oracle.offset_bias_fwd(q, k, v, bo, causal, 0.7, kv_len=kvl)
    ref = _sdpa(q, k, v, _grid(bo, n), causal, 0.7, kv_len=kvl)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bidir,causal", [(True, False), (True, True), (False, True)])
def test_alibi_is_t5_with_a_linear_table(bidir, causal):
    # 256 buckets bidirectional (128 unidirectional): 64 exact offsets per sign, so at
    # n <= 64 every offset has its own bucket and the table can hold -m |delta| exactly.
    nb = 256 if bidir else 128
    half, exact = (nb // 2, nb // 4) if bidir else (nb, nb // 2)
    B, H, n, d = 2, 3, 40, 4
    assert n - 1 < exact
    q, k, v = _inputs(B, H, n, d, 3)
    slopes = np.array([0.5, 0.125, 1.0 / 64])
    bias = np.zeros((nb, H))
    for bucket in range(nb):
        dist = bucket - half if (bidir and bucket >= half) else bucket
        bias[bucket] = -slopes * dist
    t5 = oracle.t5bias_fwd(q, k, v, bias, nb, 2 * exact, bidir, causal, 0.6)
    got = oracle.alibi_fwd(q, k, v, slopes, causal, 0.6)
    np.testing.assert_allclose(got, t5, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal,kvl", [(False, None), (True, None), (False, [5])])
def test_alibi_weights_closed_form(causal, kvl):
    # q = 0: the logit is the bias alone; v_j = e_j reads the weights out of z_i
    n, m = 7, 0.9
    q = np.zeros((1, 1, n, n))
    k = np.random.default_rng(4).standard_normal((1, 1, n, n))
    v = np.eye(n)[None, None]
    z = oracle.alibi_fwd(q, k, v, [m], causal, 1.0, kv_len=kvl)[0, 0]
    valid = n if kvl is None else kvl[0]
    for i in range(n):
        js = [j for j in range(valid) if not causal or j <= i]
        w = {j: math.exp(-m * abs(j - i)) for j in js}
        tot = sum(w.values())
        for j in range(n):
            assert abs(z[i, j] - w.get(j, 0.0) / tot) < 1e-14


def test_constant_shift_of_the_bias_changes_nothing():
    q, k, v = _inputs(1, 2, 10, 3, 5)
    bo = np.random.default_rng(6).standard_normal((2, 19))
    a = oracle.offset_bias_fwd(q, k, v, bo, True, 0.8)
    b = oracle.offset_bias_fwd(q, k, v, bo + np.array([[3.0], [-7.5]]), True, 0.8)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_clipped_table_two_token_signs():
    # offsets -1, 0, +1 get table entries a, b, c; q = k = 0 so only the bias counts
    a, b, c = -0.3, 0.4, 1.1
    q = np.zeros((1, 1, 2, 1))
    k = np.zeros((1, 1, 2, 1))
    v = np.array([0.0, 1.0]).reshape(1, 1, 2, 1)
    z = oracle.offset_table_fwd(q, k, v, [[a, b, c]], 1, False, 1.0)[0, 0, :, 0]
    # row 0: key 0 at offset 0 (b), key 1 at offset +1 (c)
    assert abs(z[0] - math.exp(c) / (math.exp(b) + math.exp(c))) < 1e-15
    # row 1: key 0 at offset -1 (a), key 1 at offset 0 (b)
    assert abs(z[1] - math.exp(b) / (math.exp(a) + math.exp(b))) < 1e-15


def test_clipped_table_radius_zero_is_plain_attention():
    q, k, v = _inputs(2, 2, 8, 3, 7)
    got = oracle.offset_table_fwd(q, k, v, [[2.5], [-1.0]], 0, False, 0.4, kv_len=[8, 5])
    ref = _sdpa(q, k, v, None, False, 0.4, kv_len=[8, 5])
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_clipped_table_clips_far_offsets_and_shares_rows():
    n, R = 12, 3
    q, k, v = _inputs(1, 2, n, 4, 8)
    table = np.random.default_rng(9).standard_normal((1, 2 * R + 1))
    bo = oracle.clipped_bias_of_offset(n, table, R, 2)
    for h in range(2):
        for delta in range(-(n - 1), n):
            assert bo[h, delta + n - 1] == table[0, max(-R, min(R, delta)) + R]
    wide = np.concatenate([np.full(n - 1 - R, table[0, 0]), table[0],
                           np.full(n - 1 - R, table[0, -1])])[None]
    np.testing.assert_array_equal(oracle.offset_table_fwd(q, k, v, table, R, False, 0.5),
                                  oracle.offset_table_fwd(q, k, v, wide, n - 1, False, 0.5))
