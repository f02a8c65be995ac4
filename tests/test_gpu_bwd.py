"""GPU parity of the gradients (relattn_bwd) against the fp64 gradient oracle
(oracle/backward.py, itself pinned to finite differences of the forward oracle).

Two paths. The SIMT kernels compute in fp32 from the exact input values (bf16 or fp32),
with the fast exponential: bar max|gpu - ref| <= 1e-3 * max|ref| + 1e-5 for every gradient.
The tensor-core kernels (bf16, d = 64 or 128) feed P, dS and the bins to the products as
bf16 with fp32 accumulation, the precision class of the bf16 forward, so they take the bf16
bar max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.
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


# cases the tensor-core kernels take (bf16, d = 64 / 128, at most 128 staged table rows),
# several query and key tiles with ragged tails among them
TC_CASES = [
    ("tiles3_bidir", 2, 2, 300, 64, 16, False, None, True, True, False, "bf16"),
    ("tiles3_causal", 2, 2, 300, 64, 16, True, None, True, True, False, "bf16"),
    ("tiles3_padded_d128", 3, 2, 260, 128, 8, False, (0, 260), True, True, False, "bf16"),
    ("causal_keyonly_k64_d128", 1, 2, 520, 128, 64, True, None, True, False, False, "bf16"),
    ("causal_k127", 1, 2, 300, 64, 127, True, None, True, True, False, "bf16"),
    ("bidir_k63_shared", 2, 2, 200, 64, 63, False, (100, 200), True, True, True, "bf16"),
    ("k0", 2, 2, 150, 64, 0, False, None, True, True, False, "bf16"),
    ("value_only_causal_d128", 2, 2, 140, 128, 16, True, (1, 140), False, True, False, "bf16"),
    ("plain_tiles", 2, 2, 257, 64, 4, False, None, False, False, False, "bf16"),
    # one query tile and one key tile per head (n <= 128, d = 64, at most 48 staged rows): the
    # one-tile kernel, at its row limit with key padding, and a single token
    ("one_tile_w47_padded", 3, 2, 128, 64, 23, False, (0, 128), True, True, False, "bf16"),
    ("one_tile_n1_causal", 2, 3, 1, 64, 4, True, None, True, True, True, "bf16"),
]


def _tc_eligible(dt, d, k, causal):
    return dt == "bf16" and d in (64, 128) and (k + 1 if causal else 2 * k + 1) <= 128


def _check(case, path, seed_extra=0):
    name, B, H, n, d, k, causal, kv, key, val, shared, dt = case
    w = wl.Workload(name, B=B, H=H, n=n, d=d, dtype=dt, clip_k=k, causal=causal,
                    kv_len_range=kv, key_term=key, value_term=val, shared_tables=shared,
                    table_std=0.5)
    x = wl.draw_inputs(w, seed=n + k + seed_extra)
    g = torch.Generator().manual_seed(n)
    dz = torch.randn((B, H, n, d), generator=g).to(w.torch_dtype)
    dev = {kk: (v.to(DEV) if v is not None else None) for kk, v in x.items()}
    rp = _rp()
    rp.relattn_set_bwd_tensor_cores(path == "tc")
    try:
        got = rp.relattn_bwd(dev["q"], dev["k"], dev["v"], dz.to(DEV), aK=dev["aK"], aV=dev["aV"],
                             clip_k=k, causal=causal, scale=w.softmax_scale, kv_len=dev["kv_len"],
                             table_head_stride=wl.table_head_stride(w))
        torch.cuda.synchronize()
    finally:
        rp.relattn_set_bwd_tensor_cores(True)
    ref = backward.relattn_bwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                               _np(dz), k, causal, w.softmax_scale,
                               kv_len=None if x["kv_len"] is None else x["kv_len"].numpy(),
                               table_head_stride=wl.table_head_stride(w))
    tc = path == "tc" and _tc_eligible(dt, d, k, causal)
    rel, ab = (1e-2, 1e-3) if tc else (1e-3, 1e-5)
    for nm, a, b in zip(("dq", "dk", "dv", "daK", "daV"), got, ref):
        if b is None:
            assert a is None
            continue
        a = a.cpu().numpy()
        tol = rel * float(np.abs(b).max()) + ab
        assert np.isfinite(a).all(), nm
        assert float(np.abs(a - b).max()) <= tol, (nm, float(np.abs(a - b).max()), tol)
    assert rp.relattn_get_device_error() == 0


@pytest.mark.parametrize("path", ["tc", "simt"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_gradients_match_oracle(case, path):
    _check(case, path)


@pytest.mark.parametrize("case", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tensor_core_gradients_match_oracle(case):
    assert _tc_eligible(case[11], case[4], case[5], case[6])
    _check(case, "tc")


@pytest.mark.parametrize("name", ["bwd_base_encoder", "bwd_big_decoder"])
def test_tensor_core_gradients_full_workload(name):
    """The gradient workloads at full size, every element of every gradient against the fp64
    oracle: bwd_base_encoder (B=64, H=8, n=128, d=64, k=16, both tables, kv_len U{32..128}:
    the one-tile kernel) and bwd_big_decoder (B=32, H=16, n=256, d=64, k=16, causal, both
    tables: the stats, keys and tables kernels over two query and two key tiles per head)."""
    w = wl.BWD_WORKLOADS[name]
    x = wl.draw_bwd_inputs(w, seed=0)
    dev = {kk: (v.to(DEV) if v is not None else None) for kk, v in x.items()}
    got = _rp().relattn_bwd(dev["q"], dev["k"], dev["v"], dev["dout"], aK=dev["aK"], aV=dev["aV"],
                            clip_k=w.clip_k, causal=w.causal, scale=w.softmax_scale,
                            kv_len=dev["kv_len"], table_head_stride=wl.table_head_stride(w))
    torch.cuda.synchronize()
    ref = backward.relattn_bwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                               _np(x["dout"]), w.clip_k, w.causal, w.softmax_scale,
                               kv_len=None if x["kv_len"] is None else x["kv_len"].numpy(),
                               table_head_stride=wl.table_head_stride(w))
    for nm, a, b in zip(("dq", "dk", "dv", "daK", "daV"), got, ref):
        a = a.cpu().numpy()
        tol = 1e-2 * float(np.abs(b).max()) + 1e-3
        assert np.isfinite(a).all(), nm
        assert float(np.abs(a - b).max()) <= tol, (nm, float(np.abs(a - b).max()), tol)
    assert _rp().relattn_get_device_error() == 0


def test_tensor_core_path_is_the_one_that_runs():
    """The default route and the SIMT route give different bits (bf16 products against fp32
    arithmetic), so an eligible call does reach the tensor-core kernels; both meet their bar."""
    B, H, n, d, k = 2, 2, 200, 64, 8
    w = wl.Workload("route", B=B, H=H, n=n, d=d, dtype="bf16", clip_k=k, table_std=0.5)
    x = wl.draw_inputs(w, seed=5)
    dz = torch.randn((B, H, n, d), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    dev = {kk: (v.to(DEV) if v is not None else None) for kk, v in x.items()}
    rp = _rp()
    outs = []
    for tc in (True, False):
        rp.relattn_set_bwd_tensor_cores(tc)
        try:
            outs.append(rp.relattn_bwd(dev["q"], dev["k"], dev["v"], dz.to(DEV), aK=dev["aK"],
                                       aV=dev["aV"], clip_k=k, scale=w.softmax_scale))
            torch.cuda.synchronize()
        finally:
            rp.relattn_set_bwd_tensor_cores(True)
    for a, b in zip(outs[0], outs[1]):
        assert not torch.equal(a, b)
        tol = 1e-2 * float(b.abs().max()) + 1e-3
        assert float((a - b).abs().max()) <= tol
    assert rp.relattn_get_device_error() == 0
