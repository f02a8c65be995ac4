"""GPU parity of relattn_labeled_bwd, the gradients of the labelled-edge forward, against the
fp64 gradient oracle (oracle/backward.py labeled_bwd, pinned to finite differences of the
labelled forward oracle and, for clip labels, to the Shaw gradients). SIMT kernels with
fp32 arithmetic from the exact inputs: max|gpu - ref| <= 1e-3 * max|ref| + 1e-5 per gradient.
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


def _f64(t):
    return None if t is None else t.double().cpu().numpy()


def _inputs(B, H, n, d, L, dtype, per_seq, shared, key, val, kv, seed):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, dz = (torch.randn((B, H, n, d), generator=g).to(tdt) for _ in range(4))
    Ht = 1 if shared else H
    aK = (torch.randn((Ht, L, d), generator=g) * 0.5).to(tdt) if key else None
    aV = (torch.randn((Ht, L, d), generator=g) * 0.5).to(tdt) if val else None
    labels = torch.randint(0, L, (B, n, n) if per_seq else (n, n), generator=g,
                           dtype=torch.int32).to(torch.uint8)
    kv_len = None if kv is None else torch.randint(kv[0], kv[1] + 1, (B,), generator=g,
                                                   dtype=torch.int32)
    return q, k, v, dz, aK, aV, labels, kv_len


@pytest.mark.parametrize("dtype,B,H,n,d,L,causal,kv,per_seq,shared,key,val", [
    ("bf16", 2, 3, 100, 64, 16, False, None, True, False, True, True),
    ("bf16", 2, 2, 150, 128, 7, True, (20, 150), False, True, True, True),
    ("f32", 2, 2, 70, 32, 256, False, (1, 70), True, False, True, True),   # every label value
    ("bf16", 1, 2, 90, 64, 9, True, None, True, False, False, True),       # value term only
    ("f32", 2, 3, 64, 48, 5, False, None, False, False, True, False),      # key term only
    ("bf16", 2, 2, 80, 64, 4, False, None, True, False, False, False),     # plain attention
])
def test_labeled_gradients_match_oracle(dtype, B, H, n, d, L, causal, kv, per_seq, shared, key,
                                        val):
    q, k, v, dz, aK, aV, labels, kv_len = _inputs(B, H, n, d, L, dtype, per_seq, shared, key,
                                                  val, kv, n + L)
    dev = lambda t: None if t is None else t.to(DEV)
    got = _rp().relattn_labeled_bwd(dev(q), dev(k), dev(v), dev(dz), dev(labels), aK=dev(aK),
                                    aV=dev(aV), num_labels=L, causal=causal, kv_len=dev(kv_len))
    torch.cuda.synchronize()
    ths = None if aK is None and aV is None else (0 if shared else L * d)
    ref = backward.labeled_bwd(_f64(q), _f64(k), _f64(v), _f64(aK), _f64(aV), _f64(dz),
                               labels.numpy(), causal, d ** -0.5,
                               kv_len=None if kv_len is None else kv_len.numpy(),
                               table_head_stride=ths)
    for nm, a, b in zip(("dq", "dk", "dv", "daK", "daV"), got, ref):
        if b is None:
            assert a is None, nm
            continue
        a = a.cpu().double().numpy()
        tol = 1e-3 * float(np.abs(b).max()) + 1e-5
        assert np.isfinite(a).all(), nm
        err = float(np.abs(a - b).max())
        assert err <= tol, (nm, err, tol)
    assert _rp().relattn_get_device_error() == 0


def test_clip_labels_give_the_shaw_gradients_bitwise():
    """Labels clip(j - i, k) + k make the labelled gradients those of relattn_bwd on its SIMT
    path: the same kernels, the same arithmetic, so the same bits."""
    rp = _rp()
    B, H, n, d, k = 2, 2, 120, 64, 6
    W = 2 * k + 1
    q, kk, v, dz, aK, aV, _, _ = _inputs(B, H, n, d, W, "bf16", False, False, True, True, None, 7)
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    labels = torch.from_numpy((np.clip(j - i, -k, k) + k).astype(np.uint8))
    args = [t.to(DEV) for t in (q, kk, v)]
    got = rp.relattn_labeled_bwd(*args, dz.to(DEV), labels.to(DEV), aK=aK.to(DEV), aV=aV.to(DEV))
    rp.relattn_set_bwd_tensor_cores(False)
    try:
        ref = rp.relattn_bwd(*args, dz.to(DEV), aK=aK.to(DEV), aV=aV.to(DEV), clip_k=k)
    finally:
        rp.relattn_set_bwd_tensor_cores(True)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert rp.relattn_get_device_error() == 0


def test_label_without_a_table_row_sets_the_status_word():
    rp = _rp()
    q, k, v, dz, aK, aV, labels, _ = _inputs(1, 2, 40, 64, 5, "bf16", False, False, True, True,
                                             None, 3)
    labels[3, 7] = 9  # no table row 9 (5 labels)
    rp.relattn_labeled_bwd(*(t.to(DEV) for t in (q, k, v, dz, labels)), aK=aK.to(DEV),
                           aV=aV.to(DEV))
    torch.cuda.synchronize()
    assert rp.relattn_get_device_error() == 1
    assert rp.relattn_get_device_error() == 0  # read and cleared
