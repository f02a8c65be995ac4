"""Pins for the fp64 gradient oracle (oracle/backward.py).

The pages give no gradients, so nothing on them can be compared directly. What fixes the
expected values here:
  * central finite differences of the forward oracle (the C triple loop in
    oracle/relattn_oracle.c, which shares no code with oracle/backward.py);
  * with zero tables, PyTorch autograd of scaled dot-product attention in float64;
  * two exact invariants of the softmax Jacobian: the value-table gradient summed over its
    rows equals the summed output gradient (sum_j p_ij = 1), and the T5 bias gradient of a
    head sums to zero over the buckets (sum_j de_ij = 0).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _fd(f, x, g, eps=1e-6):
    """Central-difference gradient of sum(f(x) * g) with respect to x (a float64 array)."""
    out = np.zeros_like(x)
    flat, of = x.reshape(-1), out.reshape(-1)
    for t in range(flat.size):
        keep = flat[t]
        flat[t] = keep + eps
        up = float((f() * g).sum())
        flat[t] = keep - eps
        dn = float((f() * g).sum())
        flat[t] = keep
        of[t] = (up - dn) / (2 * eps)
    return out


def _close(a, b, rel=1e-6):
    scale = max(float(np.abs(b).max()), 1e-12)
    assert float(np.abs(a - b).max()) <= rel * scale + 1e-9, (float(np.abs(a - b).max()), scale)


SHAW_CASES = [
    # B, H, n, d, k, causal, kv_len, with aK, with aV, shared tables
    (2, 2, 7, 3, 2, False, None, True, True, False),
    (1, 2, 6, 4, 1, True, None, True, True, False),
    (2, 1, 8, 3, 3, False, [5, 8], True, True, False),
    (1, 3, 5, 2, 2, False, None, True, True, True),
    (1, 2, 6, 3, 2, True, None, True, False, False),
    (1, 2, 6, 3, 0, False, None, False, True, False),
    (1, 1, 5, 3, 9, False, [0], True, True, False),      # a sequence with no allowed key
]


@pytest.mark.parametrize("case", SHAW_CASES)
def test_shaw_gradients_match_finite_differences(case):
    B, H, n, d, k, causal, kvl, wk, wv, shared = case
    rng = np.random.default_rng(n * 31 + d * 7 + k)
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    Ht = 1 if shared else H
    aK = rng.standard_normal((Ht, 2 * k + 1, d)) * 0.7 if wk else None
    aV = rng.standard_normal((Ht, 2 * k + 1, d)) * 0.7 if wv else None
    ths = 0 if shared else None
    kv = None if kvl is None else np.asarray(kvl, dtype=np.int32)
    scale = 0.8

    def fwd():
        return oracle.relattn_fwd(q, kk, v, aK, aV, k, causal, scale, kv_len=kv,
                                  table_head_stride=ths, nthreads=1)

    dq, dk, dv, daK, daV = backward.relattn_bwd(q, kk, v, aK, aV, dz, k, causal, scale,
                                                kv_len=kv, table_head_stride=ths)
    _close(dq, _fd(fwd, q, dz))
    _close(dk, _fd(fwd, kk, dz))
    _close(dv, _fd(fwd, v, dz))
    if wk:
        _close(daK, _fd(fwd, aK, dz))
    if wv:
        _close(daV, _fd(fwd, aV, dz))


@pytest.mark.parametrize("bidir,causal,kvl", [(True, False, None), (False, True, None),
                                              (True, False, [4, 9])])
def test_t5_gradients_match_finite_differences(bidir, causal, kvl):
    rng = np.random.default_rng(5)
    B, H, n, d = 2, 2, 9, 3
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    nb, md = 8, 6
    bias = rng.standard_normal((nb, H))
    kv = None if kvl is None else np.asarray(kvl, dtype=np.int32)
    scale = 0.6

    def fwd():
        return oracle.t5bias_fwd(q, kk, v, bias, nb, md, bidir, causal, scale, kv_len=kv,
                                 nthreads=1)

    dq, dk, dv, db = backward.t5bias_bwd(q, kk, v, bias, dz, nb, md, bidir, causal, scale,
                                         kv_len=kv)
    _close(dq, _fd(fwd, q, dz))
    _close(dk, _fd(fwd, kk, dz))
    _close(dv, _fd(fwd, v, dz))
    _close(db, _fd(fwd, bias, dz))


@pytest.mark.parametrize("causal", [False, True])
def test_zero_tables_match_torch_autograd(causal):
    rng = np.random.default_rng(11)
    B, H, n, d, k = 2, 3, 10, 4, 3
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    zeros = np.zeros((H, 2 * k + 1, d))
    scale = 0.5
    dq, dk, dv, daK, daV = backward.relattn_bwd(q, kk, v, zeros, zeros, dz, k, causal, scale)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, kk, v))
    z = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                         scale=scale)
    z.backward(torch.from_numpy(dz))
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_value_table_gradient_sums_to_output_gradient():
    """sum_r dw^V_r = sum_(i,j) p_ij dz_i = sum over rows with an allowed key of dz_i."""
    rng = np.random.default_rng(3)
    B, H, n, d, k = 2, 2, 12, 5, 2
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    aK = rng.standard_normal((H, 2 * k + 1, d)) * 0.5
    aV = rng.standard_normal((H, 2 * k + 1, d)) * 0.5
    kv = np.array([0, 7], dtype=np.int32)  # batch 0 has no allowed key at all
    _, _, _, _, daV = backward.relattn_bwd(q, kk, v, aK, aV, dz, k, False, 0.4, kv_len=kv)
    expect = dz[1].sum(axis=1)  # [H, d]: only batch 1 rows see keys
    np.testing.assert_allclose(daV.sum(axis=1), expect, rtol=1e-12, atol=1e-12)


def test_t5_bias_gradient_sums_to_zero_per_head():
    rng = np.random.default_rng(4)
    B, H, n, d = 2, 3, 20, 4
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    bias = rng.standard_normal((32, H))
    _, _, _, db = backward.t5bias_bwd(q, kk, v, bias, dz, 32, 16, True, True, 1.0)
    np.testing.assert_allclose(db.sum(axis=0), np.zeros(H), atol=1e-12)
    assert float(np.abs(db).max()) > 1e-3  # not trivially zero


@pytest.mark.parametrize("causal,kvl,per_seq", [(False, None, True), (True, None, False),
                                                (False, [3, 8], True)])
def test_labeled_gradients_match_finite_differences(causal, kvl, per_seq):
    rng = np.random.default_rng(21)
    B, H, n, d, L = 2, 2, 8, 3, 5
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    aK = rng.standard_normal((H, L, d)) * 0.7
    aV = rng.standard_normal((H, L, d)) * 0.7
    lab = rng.integers(0, L, size=(B, n, n) if per_seq else (n, n)).astype(np.uint8)
    kv = None if kvl is None else np.asarray(kvl, dtype=np.int32)

    def fwd():
        return oracle.labeled_fwd(q, kk, v, aK, aV, lab, causal, 0.8, kv_len=kv, nthreads=1)

    dq, dk, dv, daK, daV = backward.labeled_bwd(q, kk, v, aK, aV, dz, lab, causal, 0.8,
                                                kv_len=kv)
    _close(dq, _fd(fwd, q, dz))
    _close(dk, _fd(fwd, kk, dz))
    _close(dv, _fd(fwd, v, dz))
    _close(daK, _fd(fwd, aK, dz))
    _close(daV, _fd(fwd, aV, dz))


def test_labeled_gradients_with_clip_labels_are_the_shaw_gradients():
    rng = np.random.default_rng(22)
    B, H, n, d, k = 2, 2, 9, 4, 2
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    aK = rng.standard_normal((H, 2 * k + 1, d))
    aV = rng.standard_normal((H, 2 * k + 1, d))
    lab = oracle.clip_labels(n, n, k)
    got = backward.labeled_bwd(q, kk, v, aK, aV, dz, lab, True, 0.5)
    ref = backward.relattn_bwd(q, kk, v, aK, aV, dz, k, True, 0.5)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("R,shared,causal", [(2, False, False), (0, True, True), (20, False, True)])
def test_offset_table_gradients_match_finite_differences(R, shared, causal):
    rng = np.random.default_rng(23)
    B, H, n, d = 2, 2, 7, 3
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    table = rng.standard_normal((1 if shared else H, 2 * R + 1))

    def fwd():
        return oracle.offset_table_fwd(q, kk, v, table, R, causal, 0.6, nthreads=1)

    dq, dk, dv, dt = backward.offset_table_bwd(q, kk, v, table, R, dz, causal, 0.6)
    _close(dq, _fd(fwd, q, dz))
    _close(dk, _fd(fwd, kk, dz))
    _close(dv, _fd(fwd, v, dz))
    _close(dt, _fd(fwd, table, dz))


def test_alibi_gradients_match_finite_differences():
    rng = np.random.default_rng(24)
    B, H, n, d = 2, 2, 8, 3
    q, kk, v, dz = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    slopes = np.array([0.5, 0.125])

    def fwd():
        return oracle.alibi_fwd(q, kk, v, slopes, False, 0.7, kv_len=[8, 5], nthreads=1)

    dq, dk, dv, dm = backward.alibi_slope_bwd(q, kk, v, slopes, dz, False, 0.7, kv_len=[8, 5])
    _close(dq, _fd(fwd, q, dz))
    _close(dk, _fd(fwd, kk, dz))
    _close(dv, _fd(fwd, v, dz))
    _close(dm, _fd(fwd, slopes, dz))
