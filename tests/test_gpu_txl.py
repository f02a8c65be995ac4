"""GPU parity of relattn_txl_fwd (Transformer-XL relative attention) against the fp64 oracle
oracle/txl.py, on the same seeded inputs. Tolerances as elsewhere: bf16 inputs with fp32
arithmetic max|gpu - ref| <= 1e-2 * max|ref| + 1e-3; fp32 <= 1e-5 * max|ref|."""
import numpy as np
import pytest
import torch

from oracle import txl
from relative_position_representations_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _rp():
    import relative_position_representations_gb300 as rp
    return rp


def run_case(w, seed):
    rp = _rp()
    x = wl.draw_inputs(w, seed)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    got = rp.relattn_txl_fwd(g["q"], g["k"], g["v"], g["rel"], g["u"], g["vb"], causal=w.causal,
                             scale=w.softmax_scale, kv_len=g["kv_len"])
    torch.cuda.synchronize()
    f = lambda t: t.double().numpy()
    H = w.H
    rel, u, vb = f(x["rel"]), f(x["u"]), f(x["vb"])
    if rel.shape[0] == 1 and H > 1:  # one set for every head
        rel, u, vb = (np.repeat(t, H, axis=0) for t in (rel, u, vb))
    ref = txl.txl_fwd(f(x["q"]), f(x["k"]), f(x["v"]), rel, u, vb, w.causal, w.softmax_scale,
                      kv_len=None if x["kv_len"] is None else x["kv_len"].numpy())
    got = got.float().cpu().numpy()
    m = float(np.abs(ref).max())
    tol = 1e-5 * m if w.dtype == "f32" else 1e-2 * m + 1e-3
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max())
    assert err <= tol, "%s: max|err| %.3e > tol %.3e" % (w.name, err, tol)
    assert rp.relattn_get_device_error() == 0


@pytest.mark.parametrize("dtype,n,d,causal,kv,shared", [
    ("bf16", 200, 64, True, None, False),
    ("bf16", 129, 128, False, (1, 129), False),
    ("bf16", 64, 32, False, None, True),
    ("f32", 77, 32, True, (10, 77), False),
    ("f32", 50, 128, False, None, True),
    ("f32", 1, 8, True, None, False),
    # the tensor-core kernel (bf16, d = 64 / 128): several query and key tiles, ragged tails,
    # empty rows (kv_len 0), one set of encodings for all heads, a single token
    ("bf16", 300, 64, False, (0, 300), False),
    ("bf16", 385, 64, True, None, True),
    ("bf16", 257, 128, True, (100, 257), False),
    ("bf16", 1, 64, False, None, False),
    ("bf16", 130, 64, False, None, True),
])
def test_txl_matches_the_oracle(dtype, n, d, causal, kv, shared):
    w = wl.Workload("txl_case", B=2, H=3, n=n, d=d, dtype=dtype, kind="txl", causal=causal,
                    kv_len_range=kv, shared_tables=shared, table_std=0.5, qkv_std=0.7)
    run_case(w, seed=n + d)


def test_txl_decoder_workload():
    """The txl_decoder workload at full size (B=8, H=12, n=1024, d=64, causal, encodings per
    head), every output element against the oracle."""
    run_case(wl.TXL_WORKLOADS["txl_decoder"], seed=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_txl_sign_of_the_offset_matters(dtype):
    """Reversing the offset table (o -> 2n - 2 - o, i.e. j - i -> i - j) changes the output:
    the kernels (SIMT for fp32, tensor cores for bf16) read rel at j - i + n - 1, not at
    i - j + n - 1."""
    rp = _rp()
    w = wl.Workload("txl_sign", B=1, H=2, n=96, d=64, dtype=dtype, kind="txl", table_std=0.5)
    x = wl.draw_inputs(w, 11)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    a = rp.relattn_txl_fwd(g["q"], g["k"], g["v"], g["rel"], g["u"], g["vb"]).cpu()
    b = rp.relattn_txl_fwd(g["q"], g["k"], g["v"], g["rel"].flip(1).contiguous(), g["u"],
                           g["vb"]).cpu()
    assert float((a - b).abs().max()) > 1e-2


@pytest.mark.parametrize("dtype,n,dm", [("f32", 1024, 64), ("bf16", 300, 768), ("f32", 1, 2)])
def test_sinusoid_table_matches_the_oracle(dtype, n, dm):
    """relattn_sinusoid_table against the fp64 oracle table: the angle is formed in fp64, so
    the only error is the final rounding (fp32: half an ulp of values <= 1; bf16: 2^-9)."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    got = _rp().relattn_sinusoid_table(n, dm, dtype=tdt)
    torch.cuda.synchronize()
    ref = txl.sinusoid_table(n, dm)
    err = float(np.abs(got.double().cpu().numpy() - ref).max())
    assert err <= (1e-7 if dtype == "f32" else 4e-3), err


def test_txl_with_projected_sinusoids_matches_the_oracle():
    """The whole Transformer-XL position path: the library's sinusoid table, projected per head
    by W_{k,R} (a plain matrix product), as the rel argument; the oracle takes the same
    projection of its own fp64 table."""
    rp = _rp()
    B, H, n, d, dm = 2, 3, 200, 64, 96
    g = torch.Generator().manual_seed(7)
    q, k, v = (torch.randn((B, H, n, d), generator=g).to(torch.bfloat16) for _ in range(3))
    wkr = (torch.randn((H, d, dm), generator=g) * dm ** -0.5)
    u, vb = (torch.randn((H, d), generator=g).to(torch.bfloat16) for _ in range(2))
    table = rp.relattn_sinusoid_table(n, dm, dtype=torch.float32)
    rel = torch.einsum("hdm,om->hod", wkr.to(DEV), table).to(torch.bfloat16).contiguous()
    got = rp.relattn_txl_fwd(q.to(DEV), k.to(DEV), v.to(DEV), rel, u.to(DEV), vb.to(DEV),
                             causal=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    rel_ref = np.einsum("hdm,om->hod", wkr.double().numpy(), txl.sinusoid_table(n, dm))
    f = lambda t: t.double().cpu().numpy()
    ref = txl.txl_fwd(f(q), f(k), f(v), rel_ref, f(u), f(vb), True, d ** -0.5)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    assert float(np.abs(got.float().cpu().numpy() - ref).max()) <= tol
    assert rp.relattn_get_device_error() == 0
