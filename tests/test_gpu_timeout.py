"""Failure detection of the tensor-core forward on the GPU, without a fault.

Every device wait of the fused kernel is bounded. Here the bound is shortened to 10^6 SM
cycles (about half a millisecond) and the library's test hook makes each producer warp
announce the Q tiles of its first work item without loading them, so the tensor-core warp's
wait for them runs out: the kernel then takes its abort path (every role stops at its next
wait, waits for its copies and tensor-core operations in flight, frees its tensor memory and
exits). The host must read RELATTN_ERR_TIMEOUT once (the read clears it), and a normal launch
on the same context must still match the oracle. Each case runs with the short-sequence
kernel enabled and disabled (the split-feed case is the one it takes; the other two shapes
stay on the general kernel either way).
"""
import numpy as np
import pytest
import torch

import oracle
from relative_position_representations_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TIMEOUT = 4  # RELATTN_ERR_TIMEOUT

CASES = [
    # one CTA, one item: two neighbouring query tiles of one head (shared feed), d = 128,
    # key table only, causal
    wl.Workload("one_item_d128", B=1, H=1, n=256, d=128, dtype="bf16", clip_k=64,
                causal=True, value_term=False, table_std=0.5),
    # one-tile heads (split feed: two producer warps), both tables, key padding
    wl.Workload("split_feed", B=2, H=4, n=128, d=64, dtype="bf16", clip_k=16,
                table_std=0.5, kv_len_range=(40, 128)),
    # more items than CTAs (a producer meets the abort while waiting for its next item),
    # T5 scalar bias
    wl.Workload("t5_many_items", B=2, H=16, n=1024, d=64, dtype="bf16", kind="t5",
                qkv_std=0.25, scale=1.0),
]


def _rp():
    import relative_position_representations_gb300 as rp
    return rp


def _call(rp, w, g):
    if w.kind == "t5":
        return rp.relattn_t5bias_fwd(g["q"], g["k"], g["v"], g["bias"], w.num_buckets,
                                     w.max_distance, w.bidirectional, w.causal, w.softmax_scale,
                                     kv_len=g.get("kv_len"))
    return rp.relattn_fwd(g["q"], g["k"], g["v"], g["aK"], g["aV"], w.clip_k, w.causal,
                          w.softmax_scale, kv_len=g["kv_len"],
                          table_head_stride=wl.table_head_stride(w))


def _oracle(w, x):
    f = lambda t: None if t is None else t.float().numpy()
    kv = None if x.get("kv_len") is None else x["kv_len"].numpy()
    if w.kind == "t5":
        return oracle.t5bias_fwd(f(x["q"]), f(x["k"]), f(x["v"]), x["bias"].numpy(),
                                 w.num_buckets, w.max_distance, w.bidirectional, w.causal,
                                 w.softmax_scale, kv_len=kv)
    return oracle.relattn_fwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["aK"]), f(x["aV"]),
                              w.clip_k, w.causal, w.softmax_scale, kv_len=kv,
                              table_head_stride=wl.table_head_stride(w))


@pytest.mark.parametrize("short", [True, False], ids=["short_on", "short_off"])
@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_withheld_load_times_out_and_the_context_stays_usable(w, short):
    rp = _rp()
    x = wl.draw_inputs(w, seed=3)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    assert rp.relattn_get_device_error() == 0
    rp.relattn_set_wait_limit(1_000_000)
    rp.relattn_debug_withhold_first_load(True)
    rp.relattn_set_short_kernel(short)
    try:
        _call(rp, w, g)
        status = rp.relattn_get_device_error()
    finally:
        rp.relattn_set_short_kernel(True)
        rp.relattn_debug_withhold_first_load(False)
        rp.relattn_set_wait_limit(2_000_000_000)
    assert status == TIMEOUT, "expected the timeout status, got %d" % status
    assert rp.relattn_get_device_error() == 0, "the read did not clear the status word"
    # the same context, normal launches: correct output, no timeout
    for _ in range(2):
        got = _call(rp, w, g)
        torch.cuda.synchronize()
        assert rp.relattn_get_device_error() == 0
        ref = _oracle(w, x)
        err = float(np.abs(got.float().cpu().numpy() - ref).max())
        tol = 1e-2 * float(np.abs(ref).max()) + 1e-3
        assert err <= tol, "%s after the timeout: max|err| %.3e > %.3e" % (w.name, err, tol)
