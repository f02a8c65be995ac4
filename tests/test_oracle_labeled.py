"""Pins for the labelled-edge oracle (oracle.labeled_fwd).

The general form on the "Self-Attention with Relative Position Representations" page
(section "Relation-Aware Self-Attention: The Core Modification") gives every edge (i, j) of
an input graph its own a_ij; its section 3.4 specialises the edge to a table row picked by
clip(j - i, k). With an explicit label matrix L the rows are
w[L_b[i, j]]. What fixes the expected values:
  * L = clip(j - i, k) + k reproduces the Shaw forward (pinned on its own in
    test_oracle_pins.py);
  * random labels against the numpy materialised form (oracle/brute.py, which builds the
    n x n x d edge tensors and shares no code with the C loop);
  * a 2-token hand computation with asymmetric labels (catches a transposed read);
  * constant labels: the k = 0 closed forms (a constant key edge leaves the weights, a
    constant value edge is added exactly);
  * per-sequence label matrices: each sequence's rows equal a run on that sequence alone.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

RANDOM_CASES = [(False, None, False), (True, None, True), (False, [4, 11], True)]


def _inputs(B, H, n, d, seed):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((B, H, n, d)) for _ in range(3))


def test_clip_labels_reproduce_shaw():
    B, H, n, d, k = 2, 3, 13, 4, 3
    q, kk, v = _inputs(B, H, n, d, 0)
    rng = np.random.default_rng(1)
    aK = rng.standard_normal((H, 2 * k + 1, d))
    aV = rng.standard_normal((H, 2 * k + 1, d))
    lab = oracle.clip_labels(n, n, k).astype(np.uint8)
    for causal in (False, True):
        got = oracle.labeled_fwd(q, kk, v, aK, aV, lab, causal, 0.5, kv_len=[13, 6])
        ref = oracle.relattn_fwd(q, kk, v, aK, aV, k, causal, 0.5, kv_len=[13, 6])
        np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal,kvl,per_batch", RANDOM_CASES)
def test_random_labels_match_materialised_numpy(causal, kvl, per_batch):
    B, H, n, d, L = 2, 2, 11, 3, 7
    q, kk, v = _inputs(B, H, n, d, 2)
    rng = np.random.default_rng(3)
    aK = rng.standard_normal((H, L, d))
    aV = rng.standard_normal((H, L, d))
    lab = rng.integers(0, L, size=(B, n, n) if per_batch else (n, n)).astype(np.uint8)
    got = oracle.labeled_fwd(q, kk, v, aK, aV, lab, causal, 0.7, kv_len=kvl)
    ref = brute.materialised(q, kk, v, aK, aV, 0, causal, 0.7, kv_len=kvl, labels=lab,
                             num_labels=L)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_two_token_asymmetric_labels_by_hand():
    # q = 1, k = 0, v = (0, 1), key edges w^K = (0, x, y); labels [[0, 1], [2, 0]]
    x, y = 0.9, -1.7
    q = np.ones((1, 1, 2, 1))
    kk = np.zeros((1, 1, 2, 1))
    v = np.array([0.0, 1.0]).reshape(1, 1, 2, 1)
    aK = np.array([0.0, x, y]).reshape(1, 3, 1)
    lab = np.array([[0, 1], [2, 0]], dtype=np.uint8)
    z = oracle.labeled_fwd(q, kk, v, aK, None, lab, False, 1.0)[0, 0, :, 0]
    # row 0: logits 0 (key 0, label 0) and x (key 1, label 1)
    assert abs(z[0] - math.exp(x) / (1.0 + math.exp(x))) < 1e-15
    # row 1: logits y (key 0, label 2) and 0 (key 1, label 0)
    assert abs(z[1] - 1.0 / (math.exp(y) + 1.0)) < 1e-15


def test_constant_labels_closed_forms():
    B, H, n, d = 2, 2, 9, 4
    q, kk, v = _inputs(B, H, n, d, 4)
    rng = np.random.default_rng(5)
    L = 3
    aK = np.zeros((H, L, d))
    aV = np.zeros((H, L, d))
    aK[:, 2] = rng.standard_normal((H, d))
    aV[:, 2] = rng.standard_normal((H, d))
    lab = np.full((n, n), 2, dtype=np.uint8)
    got = oracle.labeled_fwd(q, kk, v, aK, aV, lab, True, 0.6)
    plain = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(kk), torch.from_numpy(v), is_causal=True,
        scale=0.6).numpy()
    np.testing.assert_allclose(got, plain + aV[None, :, 2][:, :, None, :], rtol=1e-12,
                               atol=1e-12)


def test_per_sequence_labels_are_independent():
    B, H, n, d, L = 3, 2, 8, 3, 5
    q, kk, v = _inputs(B, H, n, d, 6)
    rng = np.random.default_rng(7)
    aK = rng.standard_normal((1, L, d))
    aV = rng.standard_normal((1, L, d))
    lab = rng.integers(0, L, size=(B, n, n)).astype(np.uint8)
    full = oracle.labeled_fwd(q, kk, v, aK, aV, lab, False, 0.9, table_head_stride=0)
    for b in range(B):
        one = oracle.labeled_fwd(q[b:b + 1], kk[b:b + 1], v[b:b + 1], aK, aV, lab[b], False,
                                 0.9, table_head_stride=0)
        np.testing.assert_array_equal(full[b:b + 1], one)


def test_labels_without_a_table_row_are_refused():
    q, kk, v = _inputs(1, 1, 4, 2, 8)
    lab = np.full((4, 4), 3, dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.labeled_fwd(q, kk, v, np.zeros((1, 3, 2)), None, lab, False, 1.0)
