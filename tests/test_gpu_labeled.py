"""GPU parity of relattn_labeled_fwd (relation-aware attention over a label matrix) against
the fp64 oracle, through the C ABI.

Tolerances as elsewhere: bf16 inputs max|gpu - ref| <= 1e-2 * max|ref| + 1e-3 (here the
arithmetic is fp32, so the output rounding dominates); fp32 inputs <= 1e-5 * max|ref|.
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
    out = rp.relattn_labeled_fwd(g["q"], g["k"], g["v"], g.get("labels"), aK=g["aK"],
                                 aV=g["aV"], causal=w.causal, scale=w.softmax_scale,
                                 kv_len=g["kv_len"], table_head_stride=wl.table_head_stride(w))
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _oracle(w, x, rows=None):
    kv = None if x["kv_len"] is None else x["kv_len"].numpy()
    return oracle.labeled_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                              x["labels"].numpy(), w.causal, w.softmax_scale, kv_len=kv,
                              table_head_stride=wl.table_head_stride(w), rows=rows)


def check(w, seed=0, rows=None):
    rp = _rp()
    x = wl.draw_inputs(w, seed)
    got = _gpu(w, x)
    assert rp.relattn_get_device_error() == 0
    ref = _oracle(w, x, rows)
    if rows is not None:
        got = got.reshape(-1, w.d)[rows]
    m = float(np.abs(ref).max())
    tol = 1e-5 * m if w.dtype == "f32" else 1e-2 * m + 1e-3
    assert np.isfinite(got).all()
    err = float(np.abs(got - ref).max())
    assert err <= tol, "%s: max|err| %.3e > tol %.3e" % (w.name, err, tol)


@pytest.mark.parametrize("dtype,n,d,L,causal,kv,per_seq,shared,key,val", [
    ("bf16", 300, 64, 16, False, (40, 300), True, False, True, True),
    ("bf16", 200, 64, 7, True, None, False, True, True, True),
    ("bf16", 129, 128, 256, False, None, True, False, True, True),
    ("bf16", 70, 32, 3, False, (1, 70), True, False, True, False),
    ("bf16", 90, 64, 9, True, None, True, False, False, True),
    # the tensor-core kernel (bf16, d = 64 or 128, at most 128 labels): label rows read as
    # 16-byte vectors (n a multiple of 16) or byte by byte, several key tiles, padding, causal
    ("bf16", 512, 64, 16, False, (200, 512), True, False, True, True),
    ("bf16", 384, 128, 40, True, None, True, True, True, True),
    ("bf16", 250, 128, 128, False, (1, 250), False, False, True, True),
    ("bf16", 160, 64, 1, True, (30, 160), True, False, True, True),
    ("bf16", 256, 64, 5, False, None, False, False, False, True),
    ("bf16", 300, 128, 64, True, (100, 300), True, False, True, False),
    ("f32", 77, 32, 5, False, None, False, False, True, True),
    ("f32", 64, 128, 33, True, (10, 64), True, True, True, True),
    ("f32", 45, 20, 4, False, None, True, False, True, True),
])
def test_labeled_variants(dtype, n, d, L, causal, kv, per_seq, shared, key, val):
    w = wl.Workload("labeled_case", B=2, H=3, n=n, d=d, dtype=dtype, kind="labeled",
                    num_labels=L, causal=causal, kv_len_range=kv, labels_per_sequence=per_seq,
                    shared_tables=shared, key_term=key, value_term=val, table_std=0.5,
                    qkv_std=0.7)
    check(w, seed=n + L)


def test_clip_labels_match_the_shaw_forward():
    rp = _rp()
    B, H, n, d, k = 2, 2, 150, 64, 8
    w = wl.Workload("shaw_ref", B=B, H=H, n=n, d=d, dtype="bf16", clip_k=k, table_std=0.5)
    x = wl.draw_inputs(w, 5)
    lab = torch.from_numpy(oracle.clip_labels(n, n, k).astype(np.uint8))
    g = {key: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for key, v in x.items()}
    got = rp.relattn_labeled_fwd(g["q"], g["k"], g["v"], lab.to(DEV), aK=g["aK"], aV=g["aV"],
                                 scale=w.softmax_scale).float().cpu().numpy()
    ref = oracle.relattn_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                             k, False, w.softmax_scale)
    assert float(np.abs(got - ref).max()) <= 1e-2 * float(np.abs(ref).max()) + 1e-3


def test_no_tables_is_plain_attention():
    rp = _rp()
    q, k, v = (torch.randn(2, 2, 100, 64, generator=torch.Generator().manual_seed(s)) * 0.8
               for s in (1, 2, 3))
    got = rp.relattn_labeled_fwd(q.to(DEV), k.to(DEV), v.to(DEV), None, causal=True,
                                 scale=0.125).cpu().numpy()
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double(),
                                                           is_causal=True, scale=0.125).numpy()
    assert float(np.abs(got - ref).max()) <= 1e-5 * float(np.abs(ref).max())


def test_label_without_a_table_row_sets_the_status_word():
    # a label equal to num_labels reads the last row (in bounds) and is reported
    rp = _rp()
    w = wl.Workload("bad_label", B=1, H=2, n=40, d=64, dtype="bf16", kind="labeled",
                    num_labels=5, labels_per_sequence=False, table_std=0.5)
    x = wl.draw_inputs(w, 9)
    x["labels"][3, 7] = 5
    got = _gpu(w, x)
    assert np.isfinite(got).all()
    assert rp.relattn_get_device_error() == 1
    assert rp.relattn_get_device_error() == 0  # read and cleared
    x["labels"][3, 7] = 4
    ref = _oracle(w, x)
    assert float(np.abs(got - ref).max()) <= 1e-2 * float(np.abs(ref).max()) + 1e-3


def test_labeled_graph_workload_all_rows():
    """The labeled_graph workload at full size (B=16, H=8, n=512, d=64, 16 labels per sequence,
    both tables, kv_len U{256..512}), every output row against the oracle."""
    check(wl.LABELED_WORKLOADS["labeled_graph"], seed=1)
