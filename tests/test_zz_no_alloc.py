"""relattn_decode_fwd_noalloc (the decode step on the library's built-in device scratch)
against relattn_decode_fwd with a caller workspace of the same size, both through the C
ABI. The file name sorts last so that it runs after the other GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

from relative_position_representations_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
SCRATCH = 4 << 20  # bytes of the built-in scratch


def _lib():
    from relative_position_representations_gb300 import _lib as lib
    return lib


def _args(w, g):
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return (P(g["q"]), P(g["k"]), P(g["v"]), P(g["aK"]), P(g["aV"]),
            ctypes.c_longlong(wl.table_head_stride(w)), w.clip_k, ctypes.c_float(w.softmax_scale),
            P(g["cache_len"]), w.B, w.H, w.n, w.d)


@pytest.mark.parametrize("B,H,T", [(2, 4, 3000), (32, 16, 700)])  # split / one CTA per cache
def test_noalloc_twice_equals_workspace_call(B, H, T):
    lib = _lib()
    w = wl.Workload("noalloc", B=B, H=H, n=T, d=64, dtype="bf16", kind="decode", clip_k=16,
                    causal=True, table_std=0.5, kv_len_range=(T // 2, T))
    x = wl.draw_decode_inputs(w, seed=T)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.empty(SCRATCH, dtype=torch.uint8, device=DEV)
    ref = torch.empty_like(g["q"])
    st = lib.raw_call("relattn_decode_fwd", *_args(w, g), ctypes.c_void_p(ws.data_ptr()),
                      ctypes.c_ulonglong(SCRATCH), ctypes.c_void_p(ref.data_ptr()), stream)
    assert st == 0
    outs = []
    for _ in range(2):
        o = torch.empty_like(g["q"])
        st = lib.raw_call("relattn_decode_fwd_noalloc", *_args(w, g),
                          ctypes.c_void_p(o.data_ptr()), stream)
        assert st == 0
        outs.append(o)
    torch.cuda.synchronize()
    r = ref.float().cpu().numpy()
    for o in outs:
        assert np.array_equal(o.float().cpu().numpy(), r)
    assert np.isfinite(r).all()
    assert lib.relattn_get_device_error() == 0
