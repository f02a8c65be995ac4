"""relattn_decode_fwd_noalloc, the decode step for callers that cannot allocate device memory
(a runtime that reserves its device budget up front, a plugin handed tensors but no
allocator): it runs on a 4 MiB scratch array built into the library. Checked against
relattn_decode_fwd, both through the C ABI, on two calls in a row: with a caller workspace
of the same size when the split over the caches fits the array, and with no workspace when
the split would need more. The file name sorts last so that it runs after the other GPU
tests."""
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


@pytest.mark.parametrize("B,H,T", [(2, 4, 3000), (32, 16, 700)])  # few / many sequence-heads
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


def test_noalloc_split_larger_than_scratch_runs_unsplit():
    """8192 sequence-heads of d = 128: the split would need (1024 + 8192) records of 130
    floats (more than the 4 MiB array), so the call computes one CTA per cache like
    relattn_decode_fwd without a workspace, bit for bit. Inputs are drawn on the GPU (both
    sides are the library's own kernels; the oracle is not involved)."""
    lib = _lib()
    B, H, T, d, k = 64, 128, 384, 128, 16
    need = ctypes.c_ulonglong(0)
    assert lib.raw_call("relattn_decode_workspace_size", B, H, T, d, ctypes.byref(need)) == 0
    assert need.value > SCRATCH
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    rn = lambda *shp: torch.randn(*shp, generator=gen, device=DEV).to(torch.bfloat16)
    w = wl.Workload("noalloc_long", B=B, H=H, n=T, d=d, dtype="bf16", kind="decode",
                    clip_k=k, causal=True)
    g = {"q": rn(B, H, d), "k": rn(B, H, T, d), "v": rn(B, H, T, d),
         "aK": rn(H, 2 * k + 1, d) * 0.1, "aV": rn(H, 2 * k + 1, d) * 0.1,
         "cache_len": torch.randint(T // 2, T + 1, (B,), generator=gen, device=DEV,
                                    dtype=torch.int32)}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref = torch.empty_like(g["q"])
    st = lib.raw_call("relattn_decode_fwd", *_args(w, g), None, ctypes.c_ulonglong(0),
                      ctypes.c_void_p(ref.data_ptr()), stream)
    assert st == 0
    for _ in range(2):
        o = torch.empty_like(g["q"])
        st = lib.raw_call("relattn_decode_fwd_noalloc", *_args(w, g),
                          ctypes.c_void_p(o.data_ptr()), stream)
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(o, ref)
    assert torch.isfinite(ref.float()).all()
    assert lib.relattn_get_device_error() == 0
