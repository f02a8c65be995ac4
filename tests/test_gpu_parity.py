"""GPU parity: the CUDA library (through its C ABI) against the fp64 CPU oracle.

Inputs come from the seeded generator in workloads.py, shared by both sides. Tolerances:
bf16 inputs with fp32 accumulation, max|gpu - ref| <= 1e-2 * max|ref| + 1e-3; fp32 path
max|gpu - ref| <= 1e-5 * max|ref|; labels bit-exact.
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


def tol_for(w, ref):
    m = float(np.abs(ref).max())
    return 1e-5 * m if w.dtype == "f32" else 1e-2 * m + 1e-3


def run_gpu(w, x, stream=None):
    rp = _rp()
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    if w.kind == "t5":
        out = rp.relattn_t5bias_fwd(g["q"], g["k"], g["v"], g["bias"], w.num_buckets,
                                    w.max_distance, w.bidirectional, w.causal, w.softmax_scale,
                                    kv_len=g.get("kv_len"), stream=stream)
    else:
        out = rp.relattn_fwd(g["q"], g["k"], g["v"], g["aK"], g["aV"], w.clip_k, w.causal,
                             w.softmax_scale, kv_len=g["kv_len"],
                             table_head_stride=wl.table_head_stride(w), stream=stream)
    torch.cuda.synchronize()
    return out


def run_oracle(w, x, rows=None):
    kv = None if x.get("kv_len") is None else x["kv_len"].numpy()
    if w.kind == "t5":
        return oracle.t5bias_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), x["bias"].numpy(),
                                 w.num_buckets, w.max_distance, w.bidirectional, w.causal,
                                 w.softmax_scale, kv_len=kv, rows=rows)
    return oracle.relattn_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), _np(x["aK"]), _np(x["aV"]),
                              w.clip_k, w.causal, w.softmax_scale, kv_len=kv,
                              table_head_stride=wl.table_head_stride(w), rows=rows)


def check(w, seed=0, rows=None):
    x = wl.draw_inputs(w, seed)
    got = run_gpu(w, x).float().cpu().numpy()
    ref = run_oracle(w, x, rows)
    if rows is not None:
        got = got.reshape(-1, w.d)[rows]
    err = float(np.abs(got - ref).max())
    tol = tol_for(w, ref)
    assert np.isfinite(got).all(), "non-finite output"
    assert err <= tol, "%s: max|err| %.3e > tol %.3e" % (w.name, err, tol)
    return got, ref, err


# ------------------------------------------------------------------- fp32 SIMT path
def test_tiny_fp32_workload_full():
    check(wl.WORKLOADS["tiny_fp32"])


@pytest.mark.parametrize("n,d,k,causal,kv,shared,key,val", [
    (37, 16, 3, False, None, False, True, True),
    (64, 64, 16, True, None, False, True, True),
    (50, 33, 4, False, (1, 50), False, True, False),
    (80, 128, 70, False, (20, 80), True, True, True),
    (19, 8, 0, True, None, False, False, True),
    (23, 24, 5, False, None, False, False, False),
])
def test_fp32_variants(n, d, k, causal, kv, shared, key, val):
    w = wl.Workload("f32_case", B=3, H=2, n=n, d=d, dtype="f32", clip_k=k, causal=causal,
                    kv_len_range=kv, shared_tables=shared, key_term=key, value_term=val,
                    table_std=0.5)
    check(w, seed=n + d)


def test_fp32_t5():
    w = wl.Workload("f32_t5", B=2, H=3, n=150, d=32, dtype="f32", kind="t5", qkv_std=0.5,
                    num_buckets=32, max_distance=40)
    check(w)
    check(w.replace(bidirectional=False, causal=True), seed=1)


# ------------------------------------------------------------------- labels (S0)
@pytest.mark.parametrize("k", [0, 1, 2, 16, 64, 300])
def test_clip_labels_bit_exact(k):
    rp = _rp()
    lab = rp.relattn_labels("clip", 257, 301, clip_k=k).cpu().numpy()
    np.testing.assert_array_equal(lab, oracle.clip_labels(257, 301, k))


@pytest.mark.parametrize("nb,md,bidir", [(32, 128, True), (32, 128, False), (16, 40, True),
                                         (64, 1000, True), (8, 5, False), (4, 3, True)])
def test_t5_labels_bit_exact(nb, md, bidir):
    rp = _rp()
    n = 600
    lab = rp.relattn_labels("t5", n, n, num_buckets=nb, max_distance=md,
                            bidirectional=bidir).cpu().numpy()
    np.testing.assert_array_equal(lab, oracle.t5_labels(n, n, nb, md, bidir))


# ------------------------------------------------------------------- bf16 tensor-core path
BF16_CASES = [
    # name, n, d, k, causal, kv_len range, key term, value term, shared tables
    ("one_row", 1, 64, 2, False, None, True, True, False),
    ("ragged_37", 37, 64, 4, False, None, True, True, False),
    ("one_tile", 128, 64, 16, False, None, True, True, False),
    ("ragged_200_causal", 200, 64, 16, True, None, True, True, False),
    ("padded_300", 300, 64, 16, False, (1, 300), True, True, False),
    ("k0", 260, 64, 0, False, None, True, True, False),
    ("k1_causal", 260, 64, 1, True, None, True, True, False),
    ("k_large_causal", 390, 64, 100, True, None, True, True, False),
    ("k_over_n", 90, 64, 63, False, None, True, True, False),
    ("key_only", 517, 64, 16, True, None, True, False, False),
    ("value_only", 300, 64, 16, False, None, False, True, False),
    ("plain", 300, 64, 16, False, (100, 300), False, False, False),
    ("shared_tables", 256, 64, 8, False, None, True, True, True),
    ("d128_both", 300, 128, 16, False, (50, 300), True, True, False),
    ("d128_key_only_causal", 700, 128, 64, True, None, True, False, False),
    ("d128_k_over_n", 130, 128, 20, False, None, True, True, False),
    # one query tile per head: two heads per item on the split feed (own ring per slot)
    ("d128_one_tile_causal", 128, 128, 8, True, None, True, False, False),
    ("d128_one_tile_both", 97, 128, 8, False, (10, 97), True, True, False),
]


@pytest.mark.parametrize("case", BF16_CASES, ids=[c[0] for c in BF16_CASES])
def test_bf16_variants(case):
    w = _bf16_workload(case)
    check(w, seed=w.n + w.clip_k)


def test_bf16_one_tile_odd_head_count():
    """Five one-tile heads: the last item has a tile for one slot only (split feed)."""
    w = wl.Workload("odd_heads", B=1, H=5, n=64, d=64, dtype="bf16", clip_k=6,
                    kv_len_range=None, table_std=0.5)
    check(w, seed=3)
    check(w.replace(causal=True), seed=4)


def _bf16_workload(case):
    name, n, d, k, causal, kv, key, val, shared = case
    # large tables so that the relative terms move the output well beyond the tolerance
    return wl.Workload(name, B=2, H=3, n=n, d=d, dtype="bf16", clip_k=k, causal=causal,
                       kv_len_range=kv, key_term=key, value_term=val, shared_tables=shared,
                       table_std=0.5)


def test_bf16_relative_terms_matter_and_sign_is_checked():
    """With large tables the output differs from plain attention and from the flipped-sign
    (clip(i - j)) reading by far more than the tolerance, so parity really tests them."""
    w = wl.Workload("sign", B=2, H=2, n=300, d=64, dtype="bf16", clip_k=16, table_std=0.5)
    x = wl.draw_inputs(w, 3)
    got = run_gpu(w, x).float().cpu().numpy()
    ref = run_oracle(w, x)
    tol = tol_for(w, ref)
    assert np.abs(got - ref).max() <= tol
    flipped = oracle.relattn_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]),
                                 _np(x["aK"])[:, ::-1].copy(), _np(x["aV"])[:, ::-1].copy(),
                                 w.clip_k, False, w.softmax_scale)
    assert np.abs(got - flipped).max() > 20 * tol
    plain = oracle.relattn_fwd(_np(x["q"]), _np(x["k"]), _np(x["v"]), None, None, w.clip_k,
                               False, w.softmax_scale)
    assert np.abs(got - plain).max() > 20 * tol


@pytest.mark.parametrize("n,bidir,causal,kv", [(100, True, False, None), (300, True, False, None),
                                               (600, False, True, None),
                                               (450, True, False, (10, 450))])
def test_bf16_t5_variants(n, bidir, causal, kv):
    w = wl.Workload("t5_case", B=2, H=3, n=n, d=64, dtype="bf16", kind="t5", qkv_std=0.25,
                    scale=1.0, bidirectional=bidir, causal=causal, bias_std=2.0)
    x = wl.draw_inputs(w, n)
    if kv is not None:
        g = torch.Generator().manual_seed(5)
        x["kv_len"] = torch.randint(kv[0], kv[1] + 1, (w.B,), generator=g, dtype=torch.int32)
    got = run_gpu(w, x).float().cpu().numpy()
    ref = run_oracle(w, x)
    assert np.abs(got - ref).max() <= tol_for(w, ref)


@pytest.mark.parametrize("kind,n,d,causal,scale", [
    ("shaw", 300, 64, False, -0.125), ("shaw", 400, 128, True, -0.1), ("shaw", 300, 64, True, 0.0),
    ("t5", 300, 64, False, -0.5), ("t5", 260, 128, True, 0.0)])
def test_bf16_fused_kernel_negative_and_zero_scale(kind, n, d, causal, scale):
    """The fused kernel keeps a chunk raw (its maximum taken on the unscaled scores) only for
    a non-negative scale: a negative scale sends every chunk through the full logit, and a
    zero scale leaves only the relative terms (T5: only the bias; Shaw: uniform weights
    over the keys, the value bins still weighting the table rows). Sequences longer than
    256 keys, so the long-sequence kernel runs."""
    if kind == "t5":
        w = wl.Workload("t5_scale", B=2, H=3, n=n, d=d, dtype="bf16", kind="t5", qkv_std=0.5,
                        scale=scale, bidirectional=not causal, causal=causal, bias_std=2.0)
    else:
        w = wl.Workload("shaw_scale", B=2, H=3, n=n, d=d, dtype="bf16", clip_k=16, causal=causal,
                        table_std=0.5, scale=scale)
    check(w, seed=n + d)


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_rising_logits_force_rescales(d):
    """Logits that keep rising along the row make the running max jump by more than 2^8
    inside a key tile and across tiles, exercising the rescale of O, of the bins and of the
    P values already written for the tile."""
    w = wl.Workload("ramp_t5", B=1, H=2, n=700, d=d, dtype="bf16", kind="t5", qkv_std=0.3,
                    scale=1.0, num_buckets=32, max_distance=600)
    x = wl.draw_inputs(w, 21)
    x["bias"] = torch.zeros(32, 2)
    x["bias"][16:, :] = 2.5 * torch.arange(16, dtype=torch.float32)[:, None]
    got = run_gpu(w, x).float().cpu().numpy()
    ref = run_oracle(w, x)
    assert np.abs(got - ref).max() <= tol_for(w, ref)
    # Shaw: w^K_r = (r - k) * u with q . u > 0 on average -> rising relative logits
    kk = 60 if d == 64 else 24  # both tables at d = 128 must fit shared memory
    ws = wl.Workload("ramp_shaw", B=1, H=2, n=600, d=d, dtype="bf16", clip_k=kk,
                     table_std=0.0, kv_len_range=None)
    xs = wl.draw_inputs(ws, 22)
    u = torch.zeros(d)
    u[0] = 1.0
    xs["q"][..., 0] = 4.0
    ramp = (torch.arange(2 * kk + 1, dtype=torch.float32) - kk)[:, None] * u[None, :] * 0.8
    xs["aK"] = ramp[None].repeat(2, 1, 1).to(torch.bfloat16)
    xs["aV"] = (torch.randn(2, 2 * kk + 1, d, generator=torch.Generator().manual_seed(3)) *
                0.5).to(torch.bfloat16)
    got = run_gpu(ws, xs).float().cpu().numpy()
    ref = run_oracle(ws, xs)
    assert np.abs(got - ref).max() <= tol_for(ws, ref)


def test_bf16_t5_d128():
    w = wl.Workload("t5_d128", B=1, H=2, n=400, d=128, dtype="bf16", kind="t5", qkv_std=0.2,
                    scale=1.0, num_buckets=16, max_distance=50)
    check(w)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_shift_invariance(causal):
    """Relative-only dependence: m tokens placed at offset s inside a longer buffer give the
    same outputs as the m tokens alone. Filler keys are made unreachable through one channel
    (queries carry 1 there, real keys 0, fillers -1e4, so a filler logit is about -1e4 *
    scale and its weight underflows to exactly 0)."""
    m, s, n, d, k = 200, 131, 460, 64, 16
    w_small = wl.Workload("shift_small", B=1, H=2, n=m, d=d, dtype="bf16", clip_k=k,
                          causal=causal, table_std=0.5)
    w_big = w_small.replace(name="shift_big", n=n)
    x = wl.draw_inputs(w_small, 12)
    for name in ("q", "k", "v"):
        x[name][..., 0] = 0
    x["q"][..., 0] = 1
    x["aK"][..., 0] = 0
    big = wl.draw_inputs(w_big, 13)
    big["aK"], big["aV"] = x["aK"], x["aV"]
    big["k"][..., 0] = -1e4
    for name in ("q", "k", "v"):
        big[name][:, :, s:s + m] = x[name]
    ref = run_oracle(w_small, x)
    got_big = run_gpu(w_big, big).float().cpu().numpy()[:, :, s:s + m]
    assert np.abs(got_big - ref).max() <= tol_for(w_small, ref)


def test_bf16_deterministic_and_stream():
    w = wl.Workload("det", B=2, H=4, n=333, d=64, dtype="bf16", clip_k=16, causal=True,
                    table_std=0.5, kv_len_range=(100, 333))
    x = wl.draw_inputs(w, 4)
    a = run_gpu(w, x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run_gpu(w, x, stream=s)
    s.synchronize()
    assert torch.equal(a, b)


def test_bf16_empty_rows_are_zero():
    w = wl.Workload("empty", B=3, H=2, n=200, d=64, dtype="bf16", clip_k=4, table_std=0.5)
    x = wl.draw_inputs(w, 5)
    x["kv_len"] = torch.tensor([0, 200, 7], dtype=torch.int32)
    got = run_gpu(w, x).float().cpu().numpy()
    ref = run_oracle(w, x)
    assert (got[0] == 0).all()
    assert np.abs(got - ref).max() <= tol_for(w, ref)


def test_bf16_unsupported_and_invalid_status():
    rp = _rp()
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device=DEV)
    tab = torch.zeros(1, 129, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rp.RelattnError) as e:
        rp.relattn_fwd(q, q.clone(), q.clone(), tab, None, 64, False, 0.1)
    assert e.value.status == 2
    # both tables with 2k+1 = 127 staged rows do not fit the shared-memory budget at d = 128
    q128 = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device=DEV)
    tab127 = torch.zeros(1, 127, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rp.RelattnError) as e:
        rp.relattn_fwd(q128, q128.clone(), q128.clone(), tab127, tab127.clone(), 63, False, 0.1)
    assert e.value.status == 2
    q96 = torch.zeros(1, 1, 64, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rp.RelattnError) as e:
        rp.relattn_fwd(q96, q96.clone(), q96.clone(), None, None, 0, False, 0.1)
    assert e.value.status == 2
    assert rp.relattn_get_device_error() == 0


# ------------------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("name", ["base_encoder", "big_decoder", "long_keyonly", "t5_bias"])
def test_full_workload_all_rows(name):
    """Every output row of the full-size workload, element by element, against the oracle
    (at most a few seconds of oracle work on the host cores): every (head, query tile) of
    the launch that bench.py times is compared."""
    check(wl.WORKLOADS[name])


@pytest.mark.parametrize("name,reps", [("base_encoder", 400), ("big_decoder", 400),
                                       ("long_keyonly", 40), ("t5_bias", 80),
                                       ("ragged_200_causal", 400)])
def test_repeated_launches(name, reps):
    """Back-to-back launches on one stream: every launch gives the bitwise-same output (the
    kernel has no atomics or order-dependent sums in its data path) and no bounded device
    wait runs out. Races between the warp roles show up here as timeouts or changed outputs
    long before a single launch trips over them."""
    rp = _rp()
    if name in wl.WORKLOADS:
        w = wl.WORKLOADS[name]
    else:
        case = next(c for c in BF16_CASES if c[0] == name)
        w = _bf16_workload(case)
    x = wl.draw_inputs(w, 0)
    assert rp.relattn_get_device_error() == 0
    first = run_gpu(w, x)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    outs = []
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for r in range(reps):
            if w.kind == "t5":
                o = rp.relattn_t5bias_fwd(g["q"], g["k"], g["v"], g["bias"], w.num_buckets,
                                          w.max_distance, w.bidirectional, w.causal,
                                          w.softmax_scale, kv_len=g.get("kv_len"), stream=stream)
            else:
                o = rp.relattn_fwd(g["q"], g["k"], g["v"], g["aK"], g["aV"], w.clip_k, w.causal,
                                   w.softmax_scale, kv_len=g["kv_len"],
                                   table_head_stride=wl.table_head_stride(w), stream=stream)
            outs.append((o != first).any())
    stream.synchronize()
    assert rp.relattn_get_device_error(stream) == 0, "a device wait ran out"
    differ = int(torch.stack(outs).sum())
    assert differ == 0, "%d of %d launches differ from the first" % (differ, reps)


def test_no_device_timeouts_recorded():
    assert _rp().relattn_get_device_error() == 0
