"""GPU parity of the gradients (relattn_bwd) against the fp64 gradient oracle
(oracle/backward.py, itself pinned to finite differences of the forward oracle).

The kernels compute in fp32 from the exact input values (bf16 or fp32), with the fast
exponential, so the bar is max|gpu - ref| <= 1e-3 * max|ref| + 1e-5 for every gradient.
"""
import numpy as np
import pytest
import torch

from oracle import backward
from relative_position_representations_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _rp():
    import relative_position_representations_gb300 as rp
    return rp


def _np(t):
    return None if t is None else t.double().cpu().numpy()


CASES = [
    # name, B, H, n, d, k, causal, kv_len range, key term, value term, shared, dtype
    ("bidir", 2, 3, 100, 64, 8, False, None, True, True, False, "bf16"),
    ("causal", 2, 2, 150, 64, 16, True, None, True, True, False, "bf16"),
    ("padded", 3, 2, 90, 128, 4, False, (0, 90), True, True, False, "bf16"),
    ("shared", 2, 4, 70, 64, 8, False, None, True, True, True, "bf16"),
    ("key_only", 2, 2, 80, 64, 16, True, None, True, False, False, "bf16"),
    ("value_only", 2, 2, 80, 64, 16, False, None, False, True, False, "bf16"),
    ("plain", 2, 2, 60, 64, 3, True, None, False, False, False, "bf16"),
    ("fp32_d33", 2, 2, 50, 33, 5, False, None, True, True, False, "f32"),
    ("k_over_n", 1, 2, 40, 64, 60, False, None, True, True, False, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_gradients_match_oracle(case):
    name, B, H, n, d, k, causal, kv, key, val, shared, dt = case
    w = wl.Workload(name, B=B, H=H, n=n, d=d, dtype=dt, clip_k=k, causal=causal,
                    kv_len_range=kv, key_term=key, value_term=val, shared_tables=shared,
                    table_std=0.5)
    x = wl.draw_inputs(w, seed=n + k)
    g = torch.Generator().manual_seed(n)
    dz = torch.randn((B, H, n, d), generator=g).to(w.torch_dtype)
    dev = {kk: (v.to(DEV) if v is not None else None) for kk, v in x.items()}
    got = _rp().relattn_bwd(dev["q"], dev["k"], dev["v"], dz.to(DEV), aK=dev["aK"], aV=dev["aV"],
                            clip_k=k, causal=causal, scale=w.softmax_scale, kv_len=dev["kv_len"],
                            table_head_stride=wl.table_head_stride(w))
    torch.cuda.synchronize()
    ref = backward.relattn_bwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                               _np(dz), k, causal, w.softmax_scale,
                               kv_len=None if x["kv_len"] is None else x["kv_len"].numpy(),
                               table_head_stride=wl.table_head_stride(w))
    for nm, a, b in zip(("dq", "dk", "dv", "daK", "daV"), got, ref):
        if b is None:
            assert a is None
            continue
        a = a.cpu().numpy()
        tol = 1e-3 * float(np.abs(b).max()) + 1e-5
        assert np.isfinite(a).all(), nm
        assert float(np.abs(a - b).max()) <= tol, (nm, float(np.abs(a - b).max()), tol)
    assert _rp().relattn_get_device_error() == 0
