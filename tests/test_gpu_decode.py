"""GPU parity of the decode step (relattn_decode_fwd) against the fp64 oracle.

A decode step is row t = cache_len - 1 of the causal forward over the sequence's first
t + 1 positions, so the oracle is oracle.relattn_fwd with causal = 1, kv_len = cache_len and
the new query placed at row t (only that row is computed). Tolerance as for the bf16
forward: max|gpu - ref| <= 1e-2 * max|ref| + 1e-3.
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


def oracle_decode(w, x):
    q = x["q"].double().numpy()
    B, H, d = q.shape
    T = w.n
    lens = x["cache_len"].numpy().astype(np.int64)
    qf = np.zeros((B, H, T, d))
    rows = []
    for b in range(B):
        t = min(int(lens[b]), T) - 1
        if t < 0:
            continue
        qf[b, :, t] = q[b]
        rows += [(b * H + h) * T + t for h in range(H)]
    ref = np.zeros((B, H, d))
    if rows:
        npf = lambda t: None if t is None else t.double().numpy()
        got = oracle.relattn_fwd(qf, npf(x["k"]), npf(x["v"]), npf(x["aK"]), npf(x["aV"]),
                                 w.clip_k, True, w.softmax_scale, kv_len=lens.astype(np.int32),
                                 table_head_stride=wl.table_head_stride(w), rows=rows)
        i = 0
        for b in range(B):
            if min(int(lens[b]), T) == 0:
                continue
            for h in range(H):
                ref[b, h] = got[i]
                i += 1
    return ref


def run_decode(w, x, split=False):
    """split: pass a workspace, so the cached keys of all sequence-heads are cut into equal
    ranges, one per CTA, and merged per cache by a second kernel."""
    rp = _rp()
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    ws = None
    if split:
        nb = rp.relattn_decode_workspace_size(w.B, w.H, w.n, w.d)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
        ws.fill_(0xFF)  # scratch contents must not matter (0xFFFF... floats are NaN)
    out = rp.relattn_decode_fwd(g["q"], g["k"], g["v"], g["cache_len"], aK=g["aK"], aV=g["aV"],
                                clip_k=w.clip_k, scale=w.softmax_scale,
                                table_head_stride=wl.table_head_stride(w), workspace=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


CASES = [
    # name, B, H, T, d, k, cache lengths (None: drawn in [T/2, T]), key term, value term, shared
    ("short", 2, 3, 300, 64, 16, [300, 1], True, True, False),
    ("empty_and_full", 3, 2, 129, 64, 4, [0, 129, 64], True, True, False),
    ("chunks_d128", 2, 2, 5000, 128, 64, [5000, 2049], True, True, False),
    ("key_only", 2, 4, 700, 64, 16, None, True, False, False),
    ("value_only", 2, 4, 700, 128, 8, None, False, True, False),
    ("plain", 2, 2, 333, 64, 16, None, False, False, False),
    ("shared_tables", 2, 4, 500, 64, 16, None, True, True, True),
    ("k0", 2, 2, 200, 64, 0, None, True, True, False),
    ("k_over_len", 2, 2, 150, 64, 200, [150, 37], True, True, False),
    # fewer cached keys than CTAs of the split (CTAs without keys between a cache's pieces)
    ("tiny_total", 2, 2, 40, 64, 4, [3, 0], True, True, False),
    ("one_key", 1, 1, 8, 128, 2, [1], True, True, False),
    # many sequences of mixed lengths: ranges that start and end inside caches
    ("many_seqs", 40, 3, 257, 64, 16, None, True, True, False),
]


@pytest.mark.parametrize("split", [False, True], ids=["one_cta", "split"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(case, split):
    name, B, H, T, d, k, lens, key, val, shared = case
    w = wl.Workload(name, B=B, H=H, n=T, d=d, dtype="bf16", kind="decode", clip_k=k,
                    causal=True, key_term=key, value_term=val, shared_tables=shared,
                    table_std=0.5, kv_len_range=(max(1, T // 2), T))
    x = wl.draw_decode_inputs(w, seed=T + k)
    if lens is not None:
        x["cache_len"] = torch.tensor(lens, dtype=torch.int32)
    got = run_decode(w, x, split)
    ref = oracle_decode(w, x)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    assert np.isfinite(got).all()
    assert float(np.abs(got - ref).max()) <= tol, (float(np.abs(got - ref).max()), tol)


@pytest.mark.parametrize("split", [False, True], ids=["one_cta", "split"])
def test_decode_step_workload(split):
    w = wl.DECODE_WORKLOADS["decode_big"]
    x = wl.draw_decode_inputs(w, seed=0)
    got = run_decode(w, x, split)
    ref = oracle_decode(w, x)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    assert float(np.abs(got - ref).max()) <= tol


def test_decode_split_repeats_bitwise():
    """The split path gives the same bits on every call (no order-dependent sums)."""
    w = wl.Workload("split_rep", B=2, H=4, n=3000, d=64, dtype="bf16", kind="decode",
                    clip_k=16, causal=True, table_std=0.5, kv_len_range=(1500, 3000))
    assert _rp().relattn_decode_workspace_size(w.B, w.H, w.n, w.d) > 0
    x = wl.draw_decode_inputs(w, seed=3)
    a = run_decode(w, x, True)
    for _ in range(3):
        assert np.array_equal(run_decode(w, x, True), a)


def test_decode_relative_terms_matter():
    """With large tables the output moves well beyond the tolerance when either term is
    dropped, so the parity above really checks both."""
    w = wl.Workload("rel", B=2, H=2, n=400, d=64, dtype="bf16", kind="decode", clip_k=16,
                    causal=True, table_std=0.5, kv_len_range=(200, 400))
    x = wl.draw_decode_inputs(w, seed=9)
    got = run_decode(w, x)
    ref = oracle_decode(w, x)
    tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
    for drop in ("aK", "aV"):
        y = dict(x)
        y[drop] = torch.zeros_like(x[drop])
        alt = oracle_decode(w, y)
        assert float(np.abs(alt - ref).max()) > 5 * tol
    assert float(np.abs(got - ref).max()) <= tol
    assert _rp().relattn_get_device_error() == 0
