"""GPU parity of the short-sequence kernel (bf16 forwards with n <= 256, d = 64, at most 64
staged table rows) against the fp64 oracle, with the routing switch on (that kernel) and off
(the general fused kernel) on the same inputs.

Cases cover one and two key tiles, ragged tails (n not a multiple of 128, key padding with
zero-length sequences), causal and bidirectional rows, both tables, either table alone or
none, shared and per-head tables, k = 0, the largest staged tables (2k + 1 = 63, causal
k + 1 = 64), a negative scale (no chunk kept raw), more units than CTAs, and logits that rise
along the row so that the running maximum jumps between the two key tiles (the rescale of
O and of the bins). Tolerance: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3 elementwise.
"""
import numpy as np
import pytest
import torch

import oracle
from relative_position_representations_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _rp():
    import relative_position_representations_gb300 as rp
    return rp


def _np(t):
    return None if t is None else t.float().cpu().numpy()


def _gpu(w, x, short):
    rp = _rp()
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    rp.relattn_set_short_kernel(short)
    try:
        out = rp.relattn_fwd(g["q"], g["k"], g["v"], g["aK"], g["aV"], w.clip_k, w.causal,
                             w.softmax_scale, kv_len=g["kv_len"],
                             table_head_stride=wl.table_head_stride(w))
        torch.cuda.synchronize()
    finally:
        rp.relattn_set_short_kernel(True)
    assert rp.relattn_get_device_error() == 0
    return out.float().cpu().numpy()


def _oracle(w, x):
    kv = None if x.get("kv_len") is None else x["kv_len"].numpy()
    return oracle.relattn_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                              w.clip_k, w.causal, w.softmax_scale, kv_len=kv,
                              table_head_stride=wl.table_head_stride(w))


def _check(w, x):
    ref = _oracle(w, x)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    outs = {}
    for short in (True, False):
        got = _gpu(w, x, short)
        assert np.isfinite(got).all()
        err = float(np.abs(got - ref).max())
        assert err <= tol, "%s (short=%s): max|err| %.3e > %.3e" % (w.name, short, err, tol)
        outs[short] = got
    return outs


CASES = [
    # name, B, H, n, k, causal, kv_len range, shared tables, key table, value table
    ("one_tile_both", 2, 3, 128, 16, False, None, False, True, True),
    ("ragged_100", 2, 2, 100, 16, False, None, False, True, True),
    ("two_tiles_causal", 2, 4, 256, 16, True, None, False, True, True),
    ("two_tiles_bidir_padded", 3, 2, 256, 16, False, (0, 256), False, True, True),
    ("ragged_200_causal", 2, 2, 200, 8, True, (1, 200), True, True, True),
    ("tiny_n", 2, 2, 7, 3, False, None, False, True, True),
    ("n_129", 1, 3, 129, 16, True, None, False, True, True),
    ("key_only", 2, 2, 160, 16, False, (20, 160), False, True, False),
    ("value_only", 2, 2, 160, 16, True, None, False, False, True),
    ("no_tables", 2, 2, 192, 4, False, (33, 192), False, False, False),
    ("k0", 2, 2, 128, 0, False, None, False, True, True),
    ("k_over_n", 1, 2, 40, 31, False, None, False, True, True),
    ("w63_bidir", 2, 2, 256, 31, False, (100, 256), False, True, True),
    ("w64_causal", 2, 2, 256, 63, True, None, True, True, True),
    ("many_units", 8, 48, 256, 16, True, None, False, True, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_short_kernel_matches_oracle(case):
    name, B, H, n, k, causal, kv, shared, key, val = case
    w = wl.Workload(name, B=B, H=H, n=n, d=64, dtype="bf16", clip_k=k, causal=causal,
                    kv_len_range=kv, shared_tables=shared, key_term=key, value_term=val,
                    table_std=0.5)
    _check(w, wl.draw_inputs(w, seed=n + k))


def test_short_kernel_negative_scale():
    """A negative scale keeps no chunk raw (the raw path needs max(x * s) = s * max(x))."""
    w = wl.Workload("neg_scale", B=2, H=2, n=256, d=64, dtype="bf16", clip_k=16, causal=False,
                    table_std=0.5, kv_len_range=(50, 256), scale=-0.125)
    _check(w, wl.draw_inputs(w, seed=5))


def test_short_kernel_rising_logits_rescale():
    """w^K_r = (r - k) u with q . u large: the logits rise along the row, so the second key
    tile's maximum exceeds the first by more than 2^8 and O and the bins are rescaled."""
    kk = 31
    w = wl.Workload("ramp_short", B=1, H=2, n=256, d=64, dtype="bf16", clip_k=kk, table_std=0.0)
    x = wl.draw_inputs(w, 22)
    u = torch.zeros(64)
    u[0] = 1.0
    x["q"][..., 0] = 4.0
    ramp = (torch.arange(2 * kk + 1, dtype=torch.float32) - kk)[:, None] * u[None, :] * 0.8
    x["aK"] = ramp[None].repeat(2, 1, 1).to(torch.bfloat16)
    x["aV"] = (torch.randn(2, 2 * kk + 1, 64, generator=torch.Generator().manual_seed(3)) *
               0.5).to(torch.bfloat16)
    # keys placed so that a far-right block of keys beats the first tile's best logit
    x["k"][..., 128:, 0] = 3.0
    _check(w, x)


@pytest.mark.parametrize("name", ["base_encoder", "big_decoder"])
def test_short_kernel_full_workload_both_paths_agree(name):
    """The workloads this kernel serves, every output row, on both kernels."""
    w = wl.WORKLOADS[name]
    _check(w, wl.draw_inputs(w, seed=0))


def test_short_kernel_repeated_launches_bitwise():
    w = wl.WORKLOADS["big_decoder"]
    x = wl.draw_inputs(w, seed=1)
    rp = _rp()
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    outs = []
    for _ in range(60):
        outs.append(rp.relattn_fwd(g["q"], g["k"], g["v"], g["aK"], g["aV"], w.clip_k, w.causal,
                                   w.softmax_scale, kv_len=g["kv_len"],
                                   table_head_stride=wl.table_head_stride(w)))
    torch.cuda.synchronize()
    assert rp.relattn_get_device_error() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
