"""GPU parity of the scalar offset biases (ALiBi and the clipped per-offset table) against
the fp64 oracle, through the C ABI.

Both ride on the T5 form of the fused kernel ("Relative position embeddings" page,
sections "T5" and "Placement in the taxonomy"): only the shared-memory table of biases over
the offsets is filled differently. Tolerances as in test_gpu_parity.py: bf16
max|gpu - ref| <= 1e-2 * max|ref| + 1e-3, fp32 <= 1e-5 * max|ref|.
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


def _gpu(w, x):
    rp = _rp()
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    if w.kind == "alibi":
        out = rp.relattn_alibi_fwd(g["q"], g["k"], g["v"], g["slopes"], w.causal,
                                   w.softmax_scale, kv_len=g["kv_len"])
    else:
        out = rp.relattn_offset_bias_fwd(g["q"], g["k"], g["v"], g["table"], w.clip_k, w.causal,
                                         w.softmax_scale, kv_len=g["kv_len"])
    torch.cuda.synchronize()
    assert rp.relattn_get_device_error() == 0
    return out.float().cpu().numpy()


def _oracle(w, x, rows=None):
    kv = None if x["kv_len"] is None else x["kv_len"].numpy()
    if w.kind == "alibi":
        return oracle.alibi_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), x["slopes"].numpy(),
                                w.causal, w.softmax_scale, kv_len=kv, rows=rows)
    return oracle.offset_table_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), x["table"].numpy(),
                                   w.clip_k, w.causal, w.softmax_scale, kv_len=kv, rows=rows)


def check(w, seed=0, rows=None):
    x = wl.draw_inputs(w, seed)
    got = _gpu(w, x)
    ref = _oracle(w, x, rows)
    if rows is not None:
        got = got.reshape(-1, w.d)[rows]
    m = float(np.abs(ref).max())
    tol = 1e-5 * m if w.dtype == "f32" else 1e-2 * m + 1e-3
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max())
    assert err <= tol, "%s: max|err| %.3e > tol %.3e" % (w.name, err, tol)
    return got, ref


@pytest.mark.parametrize("n,d,causal,kv,max_bias", [
    (300, 64, True, None, 8.0),
    (100, 64, False, (1, 100), 8.0),
    (64, 64, False, None, 2.0),          # one query tile per head
    (700, 128, False, None, 2.0),
    (257, 128, True, None, 8.0),         # two full tiles and one row
])
def test_bf16_alibi(n, d, causal, kv, max_bias):
    w = wl.Workload("alibi_case", B=2, H=3, n=n, d=d, dtype="bf16", kind="alibi",
                    causal=causal, kv_len_range=kv, alibi_max_bias=max_bias)
    check(w, seed=n + d)


def test_bf16_alibi_bias_decides_the_output():
    # with these slopes the bias dominates the content term: a sign or offset slip in the
    # kernel's table moves the output by far more than the tolerance
    w = wl.Workload("alibi_strong", B=1, H=2, n=200, d=64, dtype="bf16", kind="alibi",
                    causal=False, qkv_std=0.3, alibi_max_bias=1.0)
    x = wl.draw_inputs(w, 3)
    got = _gpu(w, x)
    ref = _oracle(w, x)
    plain = oracle.alibi_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), np.zeros(2), False,
                             w.softmax_scale)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    assert float(np.abs(got - ref).max()) <= tol
    assert float(np.abs(plain - ref).max()) > 5 * tol


def test_bf16_alibi_long_sequence_sampled_rows():
    # the whole offset range of a 2048-token sequence in shared memory
    w = wl.Workload("alibi_long", B=1, H=2, n=2048, d=64, dtype="bf16", kind="alibi",
                    causal=True)
    rows = np.random.default_rng(0).choice(w.H * w.n, size=256, replace=False)
    rows = np.sort(np.concatenate([rows, [0, w.n - 1, w.n, 2 * w.n - 1]]))
    check(w, seed=11, rows=np.unique(rows))


@pytest.mark.parametrize("n,d,R,causal,shared,kv", [
    (300, 64, 0, False, False, None),
    (300, 64, 5, True, False, None),
    (200, 64, 40, False, True, (30, 200)),
    (150, 64, 1000, False, False, None),  # radius beyond the sequence: no clipping
    (257, 128, 17, True, True, None),
    (64, 128, 128, False, False, (1, 64)),
])
def test_bf16_offset_table(n, d, R, causal, shared, kv):
    w = wl.Workload("offset_case", B=2, H=3, n=n, d=d, dtype="bf16", kind="offset", clip_k=R,
                    causal=causal, shared_tables=shared, kv_len_range=kv, bias_std=1.5)
    check(w, seed=n + R)


@pytest.mark.parametrize("kind,n,d,causal,R,kv", [
    ("alibi", 50, 32, True, 0, None),
    ("alibi", 37, 16, False, 0, (1, 37)),
    ("offset", 40, 16, False, 3, (5, 40)),
    ("offset", 33, 64, True, 50, None),
])
def test_fp32_scalar_biases(kind, n, d, causal, R, kv):
    w = wl.Workload("f32_bias", B=2, H=2, n=n, d=d, dtype="f32", kind=kind, clip_k=R,
                    causal=causal, kv_len_range=kv, alibi_max_bias=4.0, qkv_std=0.5)
    check(w, seed=n)


def test_bf16_alibi_too_long_for_shared_memory_is_unsupported():
    # the bias of every offset does not fit shared memory: refused on the host, no launch
    rp = _rp()
    n = 40000
    q = torch.zeros((1, 1, n, 64), dtype=torch.bfloat16, device=DEV)
    slopes = torch.ones(1, dtype=torch.float32, device=DEV)
    with pytest.raises(rp.RelattnError) as e:
        rp.relattn_alibi_fwd(q, q.clone(), q.clone(), slopes, causal=True)
    assert e.value.status == 2


@pytest.mark.parametrize("name", ["alibi_decoder", "offset_bias"])
def test_bias_workload_all_rows(name):
    """The scalar-bias workloads at full size (B=8, H=12, n=2048, d=64: ALiBi in a causal
    decoder, a per-head offset table clipped at 128 in a bidirectional encoder), every output
    row against the oracle, as bench.py times them."""
    check(wl.BIAS_WORKLOADS[name], seed=0)
