"""GPU parity of relattn_scalar_bias_bwd, the gradients of the T5, ALiBi and per-offset-table
forwards, against the fp64 gradient oracles (oracle/backward.py: t5bias_bwd, alibi_slope_bwd,
offset_table_bwd, themselves pinned to finite differences of the forward oracles).

The kernels compute in fp32 from the exact input values (bf16 or fp32) on the SIMT units,
with the fast exponential, so they take the SIMT gradient bar of relattn_bwd:
max|gpu - ref| <= 1e-3 * max|ref| + 1e-5 for every output, the parameter's gradient included.
"""
import numpy as np
import pytest
import torch

from oracle import backward

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _rp():
    import relative_position_representations_gb300 as rp
    return rp


def _draw(B, H, n, d, dtype, seed, kv):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, dz = (torch.randn((B, H, n, d), generator=g).to(tdt) for _ in range(4))
    kv_len = None
    if kv is not None:
        kv_len = torch.randint(kv[0], kv[1] + 1, (B,), generator=g, dtype=torch.int32)
    return q, k, v, dz, kv_len


def _compare(got, ref):
    for nm, a, b in zip(("dq", "dk", "dv", "dbias"), got, ref):
        a = a.cpu().double().numpy()
        b = np.asarray(b, dtype=np.float64).reshape(a.shape)
        tol = 1e-3 * float(np.abs(b).max()) + 1e-5
        assert np.isfinite(a).all(), nm
        err = float(np.abs(a - b).max())
        assert err <= tol, (nm, err, tol)


def _f64(t):
    return None if t is None else t.double().numpy()


@pytest.mark.parametrize("dtype,B,H,n,d,nb,md,bidir,causal,kv", [
    ("bf16", 2, 3, 100, 64, 32, 128, True, False, None),
    ("bf16", 2, 2, 300, 64, 32, 128, False, True, None),     # unidirectional T5, causal decoder
    ("f32", 3, 2, 77, 32, 16, 50, True, False, (1, 77)),     # padded keys, other d
    ("bf16", 1, 2, 260, 128, 8, 20, True, True, (100, 260)),
])
def test_t5_bias_gradients(dtype, B, H, n, d, nb, md, bidir, causal, kv):
    q, k, v, dz, kv_len = _draw(B, H, n, d, dtype, n + nb, kv)
    bias = torch.randn((nb, H), generator=torch.Generator().manual_seed(nb)) * 2.0
    got = _rp().relattn_scalar_bias_bwd(q.to(DEV), k.to(DEV), v.to(DEV), dz.to(DEV), "t5",
                                        bias.to(DEV), num_buckets=nb, max_distance=md,
                                        bidirectional=bidir, causal=causal, scale=0.5,
                                        kv_len=None if kv_len is None else kv_len.to(DEV))
    torch.cuda.synchronize()
    ref = backward.t5bias_bwd(_f64(q), _f64(k), _f64(v), bias.double().numpy(), _f64(dz), nb, md,
                              bidir, causal, 0.5,
                              kv_len=None if kv_len is None else kv_len.numpy())
    _compare(got, ref)
    assert _rp().relattn_get_device_error() == 0


@pytest.mark.parametrize("dtype,B,H,n,d,causal,kv", [
    ("bf16", 2, 4, 200, 64, True, None),
    ("f32", 2, 2, 90, 48, False, (10, 90)),
    ("bf16", 1, 3, 513, 128, False, None),
])
def test_alibi_slope_gradients(dtype, B, H, n, d, causal, kv):
    q, k, v, dz, kv_len = _draw(B, H, n, d, dtype, n + d, kv)
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32)
    got = _rp().relattn_scalar_bias_bwd(q.to(DEV), k.to(DEV), v.to(DEV), dz.to(DEV), "alibi",
                                        slopes.to(DEV), causal=causal,
                                        kv_len=None if kv_len is None else kv_len.to(DEV))
    torch.cuda.synchronize()
    ref = backward.alibi_slope_bwd(_f64(q), _f64(k), _f64(v), slopes.double().numpy(), _f64(dz),
                                   causal, d ** -0.5,
                                   kv_len=None if kv_len is None else kv_len.numpy())
    _compare(got, ref)
    assert _rp().relattn_get_device_error() == 0


@pytest.mark.parametrize("dtype,B,H,n,d,R,shared,causal,kv", [
    ("bf16", 2, 3, 150, 64, 8, False, False, None),
    ("bf16", 2, 3, 150, 64, 8, True, True, None),             # one row for every head
    ("f32", 2, 2, 60, 32, 1000, False, False, (5, 60)),       # radius beyond the sequence
    ("bf16", 1, 2, 300, 128, 2, True, False, None),
])
def test_offset_table_gradients(dtype, B, H, n, d, R, shared, causal, kv):
    q, k, v, dz, kv_len = _draw(B, H, n, d, dtype, n + R, kv)
    table = torch.randn((1 if shared else H, 2 * R + 1), generator=torch.Generator().manual_seed(R))
    got = _rp().relattn_scalar_bias_bwd(q.to(DEV), k.to(DEV), v.to(DEV), dz.to(DEV), "table",
                                        table.to(DEV), radius=R, causal=causal,
                                        kv_len=None if kv_len is None else kv_len.to(DEV))
    torch.cuda.synchronize()
    ref = backward.offset_table_bwd(_f64(q), _f64(k), _f64(v), table.double().numpy(), R,
                                    _f64(dz), causal, d ** -0.5,
                                    kv_len=None if kv_len is None else kv_len.numpy())
    _compare(got, ref)
    assert _rp().relattn_get_device_error() == 0


def test_bias_gradient_sees_the_offset_sign():
    """Flipping the table (offset o -> -o) changes the output's gradient with respect to the
    table by far more than the tolerance: the kernels index the bias by j - i, not i - j."""
    q, k, v, dz, _ = _draw(1, 2, 64, 64, "bf16", 5, None)
    R = 6
    table = torch.randn((2, 2 * R + 1), generator=torch.Generator().manual_seed(9)) * 3.0
    rp = _rp()
    args = [t.to(DEV) for t in (q, k, v, dz)]
    a = rp.relattn_scalar_bias_bwd(*args, "table", table.to(DEV), radius=R, causal=False)[3]
    b = rp.relattn_scalar_bias_bwd(*args, "table", table.flip(1).contiguous().to(DEV), radius=R,
                                   causal=False)[3]
    ref = backward.offset_table_bwd(_f64(q), _f64(k), _f64(v), table.double().numpy(), R,
                                    _f64(dz), False, 64 ** -0.5)[3]
    tol = 1e-3 * float(np.abs(ref).max()) + 1e-5
    assert float(np.abs(a.cpu().double().numpy() - ref).max()) <= tol
    assert float(np.abs(b.cpu().double().numpy() - ref).max()) > 20 * tol


def test_constant_bias_has_zero_gradient():
    """Radius 0: one scalar added to every logit of every head. The softmax is invariant to
    it, so its exact gradient is 0 (each row's de sums to 0) while dq, dk, dv are those of
    plain attention. The device sum of ~180K cancelling fp32 terms stays within 1e-4 of
    their L1 mass (computed here in fp64 from the same inputs)."""
    B, H, n, d = 1, 2, 300, 128
    q, k, v, dz, _ = _draw(B, H, n, d, "bf16", 300, None)
    table = torch.tensor([[0.7]])
    got = _rp().relattn_scalar_bias_bwd(q.to(DEV), k.to(DEV), v.to(DEV), dz.to(DEV), "table",
                                        table.to(DEV), radius=0, causal=False)
    torch.cuda.synchronize()
    ref = backward.offset_table_bwd(_f64(q), _f64(k), _f64(v), table.double().numpy(), 0,
                                    _f64(dz), False, d ** -0.5)
    _compare(got[:3], ref[:3])
    l1 = 0.0
    for h in range(H):
        qh, kh, vh, gz = (_f64(t)[0, h] for t in (q, k, v, dz))
        e = d ** -0.5 * (qh @ kh.T)
        p = np.exp(e - e.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dp = gz @ vh.T
        l1 += float(np.abs(p * (dp - (p * dp).sum(axis=1, keepdims=True))).sum())
    assert abs(float(got[3].item())) <= 1e-4 * l1
    assert _rp().relattn_get_device_error() == 0
