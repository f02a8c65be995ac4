"""The C-ABI library: it builds, loads, exports every symbol include/relattn.h declares,
and its host-only logic is right. No kernel is launched here (these run without a GPU):
invalid arguments are rejected before any CUDA call, and the exact T5 thresholds come from
host code."""
import ctypes
import os
import re

import pytest

import oracle
from oracle import t5 as ot5

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from relative_position_representations_gb300 import build
    build.build()
    from relative_position_representations_gb300 import _lib
    return _lib


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "relattn.h")).read()
    return sorted(set(re.findall(r"RELATTN_API\s+[\w\s\*]+?\b(relattn_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for want in ("relattn_fwd", "relattn_t5bias_fwd", "relattn_labels", "relattn_t5_thresholds",
                 "relattn_get_device_error", "relattn_status_string", "relattn_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(so, name), name
    assert sorted(lib.EXPORTED) == sorted(declared_symbols())


def test_status_strings_and_version(lib):
    assert lib.relattn_version() >= 100
    assert lib.relattn_status_string(0) == "ok"
    assert "timed out" in lib.relattn_status_string(4)
    assert lib.relattn_status_string(99) == "unknown status"


def test_wait_limit_and_hook_arguments_checked_on_the_host(lib):
    """Host-only checks of the failure-detection settings (no launch)."""
    assert lib.raw_call("relattn_set_wait_limit", 10) == 1  # below 1000 cycles
    assert lib.raw_call("relattn_set_wait_limit", 1 << 41) == 1
    assert lib.raw_call("relattn_debug_withhold_first_load", 2) == 1
    assert lib.raw_call("relattn_set_wait_limit", 2000000000) == 0  # the default
    assert lib.raw_call("relattn_debug_withhold_first_load", 0) == 0
    assert lib.raw_call("relattn_set_short_kernel", 2) == 1
    assert lib.raw_call("relattn_set_short_kernel", 0) == 0
    assert lib.raw_call("relattn_set_short_kernel", 1) == 0  # the default
    assert lib.raw_call("relattn_set_bwd_tensor_cores", 2) == 1
    assert lib.raw_call("relattn_set_bwd_tensor_cores", 0) == 0
    assert lib.raw_call("relattn_set_bwd_tensor_cores", 1) == 0  # the default
    # sinusoid table: a null output, an odd d_model and a bad dtype are refused on the host
    assert lib.raw_call("relattn_sinusoid_table", 4, 8, 0, None, None) == 1
    # (a pointer value that the host check rejects first, never dereferenced)
    assert lib.raw_call("relattn_sinusoid_table", 4, 7, 0, 256, None) == 1
    assert lib.raw_call("relattn_sinusoid_table", 4, 8, 7, 256, None) == 1


@pytest.mark.parametrize("nb,md,bidir", [(32, 128, True), (32, 128, False), (16, 40, True),
                                         (64, 1000, True), (8, 5, False), (4, 3, True),
                                         (256, 100000, True), (200, 7000, False)])
def test_host_t5_thresholds_match_oracle_buckets(lib, nb, md, bidir):
    thr = lib.relattn_t5_thresholds(nb, md, bidir)
    half = nb // 2 if bidir else nb
    exact = half // 2
    assert len(thr) == half - 1 - exact
    sign = -1  # lower half (offsets <= 0)
    for m, a in enumerate(thr):
        b = exact + 1 + m
        assert ot5.t5_bucket(sign * a, nb, md, bidir) >= b
        assert ot5.t5_bucket(sign * (a - 1), nb, md, bidir) < b


def test_default_thresholds_are_the_closed_form_values(lib):
    assert lib.relattn_t5_thresholds(32, 128, True) == [12, 16, 23, 32, 46, 64, 91]


FAKE = ctypes.c_void_p(0x100000)  # aligned, never dereferenced on the host


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, aK=None, aV=None, ths=0, clip_k=2, causal=0, scale=1.0,
         kv=None, B=1, H=1, n=16, d=64, dtype=0, out=ctypes.c_void_p(0x200000)):
    return lib.raw_call("relattn_fwd", q, k, v, aK, aV, ctypes.c_longlong(ths), clip_k, causal,
                        ctypes.c_float(scale), kv, B, H, n, d, dtype, out, None)


def test_invalid_arguments_rejected_before_any_launch(lib):
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, out=FAKE) == 1                      # aliases q
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, clip_k=-1) == 1
    assert _fwd(lib, causal=2) == 1
    assert _fwd(lib, dtype=7) == 1
    assert _fwd(lib, q=ctypes.c_void_p(0x100008)) == 1   # bf16 needs 16-byte alignment
    assert _fwd(lib, d=96) == 2                          # bf16 head dims: 64 and 128
    assert _fwd(lib, dtype=1, d=200) == 2                # fp32 path: d <= 128
    assert _fwd(lib, aK=ctypes.c_void_p(0x300000), ths=10) == 1   # stride below the table
    bad_t5 = lib.raw_call("relattn_t5bias_fwd", FAKE, FAKE, FAKE, ctypes.c_void_p(0x300000), 2,
                          128, 1, 0, ctypes.c_float(1.0), None, 1, 1, 16, 64, 0,
                          ctypes.c_void_p(0x200000), None)
    assert bad_t5 == 1                                   # 2 buckets bidirectional: no exact range
    bad_t5 = lib.raw_call("relattn_t5bias_fwd", FAKE, FAKE, FAKE, ctypes.c_void_p(0x300000), 32,
                          8, 1, 0, ctypes.c_float(1.0), None, 1, 1, 16, 64, 0,
                          ctypes.c_void_p(0x200000), None)
    assert bad_t5 == 1                                   # max_distance inside the exact range
    assert lib.raw_call("relattn_labels", 5, 0, 32, 128, 1, 4, 4, FAKE, None) == 1


def test_offset_bias_arguments_rejected_before_any_launch(lib):
    TAB = ctypes.c_void_p(0x300000)
    OUT = ctypes.c_void_p(0x200000)

    def offs(table=TAB, ths=0, radius=4, causal=0, dtype=0, d=64):
        return lib.raw_call("relattn_offset_bias_fwd", FAKE, FAKE, FAKE, table,
                            ctypes.c_longlong(ths), radius, causal, ctypes.c_float(1.0), None,
                            1, 2, 16, d, dtype, OUT, None)

    def alibi(slopes=TAB, causal=0, d=64):
        return lib.raw_call("relattn_alibi_fwd", FAKE, FAKE, FAKE, slopes, causal,
                            ctypes.c_float(1.0), None, 1, 2, 16, d, 0, OUT, None)

    assert offs(radius=-1) == 1
    assert offs(radius=(1 << 20) + 1) == 1
    assert offs(ths=5) == 1                               # head stride below 2*radius + 1
    assert offs(table=None) == 1
    assert offs(table=ctypes.c_void_p(0x300002)) == 1      # fp32 table: 4-byte alignment
    assert offs(causal=3) == 1
    assert offs(d=96) == 2
    assert alibi(slopes=None) == 1
    assert alibi(causal=-1) == 1
    assert alibi(d=32) == 2


def test_labeled_arguments_rejected_before_any_launch(lib):
    TAB = ctypes.c_void_p(0x300000)
    LAB = ctypes.c_void_p(0x400000)
    OUT = ctypes.c_void_p(0x200000)

    def lab(aK=TAB, aV=None, ths=0, L=8, labels=LAB, lbs=0, causal=0, n=16, d=64, dtype=0):
        return lib.raw_call("relattn_labeled_fwd", FAKE, FAKE, FAKE, aK, aV,
                            ctypes.c_longlong(ths), L, labels, ctypes.c_longlong(lbs), causal,
                            ctypes.c_float(1.0), None, 1, 2, n, d, dtype, OUT, None)

    assert lab(L=0) == 1
    assert lab(L=257) == 1
    assert lab(labels=None) == 1
    assert lab(lbs=100) == 1                       # below n * n
    assert lab(ths=8 * 64 - 8) == 1                # below num_labels * d
    assert lab(ths=8 * 64 + 4) == 1                # bf16 rows: a multiple of 8 elements
    assert lab(aK=ctypes.c_void_p(0x300008)) == 1  # tables 16-byte aligned
    assert lab(causal=2) == 1
    assert lab(d=36) == 2                          # bf16: d a multiple of 8
    assert lab(d=136) == 2
    assert lab(dtype=1, d=130) == 2


def test_scalar_bias_bwd_arguments_rejected_before_any_launch(lib):
    BIAS = ctypes.c_void_p(0x300000)
    WS = ctypes.c_void_p(0x400000)
    G = [ctypes.c_void_p(0x500000 + i * 0x100000) for i in range(4)]  # dq, dk, dv, dbias

    def call(kind=1, bias=BIAS, nb=32, md=128, bidir=1, radius=4, hs=0, causal=0, n=16, d=64,
             dtype=0, dout=FAKE, ws=WS, wsb=1 << 30):
        return lib.raw_call("relattn_scalar_bias_bwd", FAKE, FAKE, FAKE, dout, kind, bias, nb, md,
                            bidir, radius, ctypes.c_longlong(hs), causal, ctypes.c_float(1.0), None,
                            1, 2, n, d, dtype, G[0], G[1], G[2], G[3], ws, ctypes.c_ulonglong(wsb),
                            None)

    assert call(kind=3) == 1
    assert call(kind=-1) == 1
    assert call(bias=None) == 1
    assert call(bias=ctypes.c_void_p(0x300002)) == 1      # fp32 parameters: 4-byte alignment
    assert call(dout=None) == 1
    assert call(ws=None) == 1
    assert call(kind=0, nb=1) == 1                         # no valid bucket layout
    assert call(kind=0, bidir=2) == 1
    assert call(kind=2, radius=-1) == 1
    assert call(kind=2, radius=4, hs=5) == 1               # head stride below 2*radius + 1
    assert call(causal=2) == 1
    assert call(wsb=16) == 1                               # workspace below the size query
    assert call(n=4097) == 2                               # beyond the shared-memory offset rows
    assert lib.raw_call("relattn_scalar_bias_bwd", FAKE, FAKE, FAKE, FAKE, 1, BIAS, 32, 128, 1, 4,
                        ctypes.c_longlong(0), 0, ctypes.c_float(1.0), None, 256, 257, 16, 64, 0,
                        G[0], G[1], G[2], G[3], WS, ctypes.c_ulonglong(1 << 40), None) == 2
    assert call(d=256, dtype=1) == 2
    nb = ctypes.c_ulonglong(0)
    assert lib.raw_call("relattn_scalar_bias_bwd_workspace_size", 2, 3, 5, ctypes.byref(nb)) == 0
    # per-row records (3 floats for each of the 30 rows, rounded up to a multiple of 64) and
    # the per-offset sums of every head (3 heads x 9 offsets)
    assert nb.value == (128 + 3 * (2 * 5 - 1)) * 4


def test_labeled_bwd_arguments_rejected_before_any_launch(lib):
    TAB = ctypes.c_void_p(0x300000)
    LAB = ctypes.c_void_p(0x380000)
    WS = ctypes.c_void_p(0x400000)
    G = [ctypes.c_void_p(0x500000 + i * 0x100000) for i in range(5)]  # dq, dk, dv, daK, daV

    def call(aK=TAB, aV=None, ths=0, L=8, labels=LAB, lbs=0, causal=0, n=16, d=64, dtype=0,
             daK=G[3], daV=G[4], ws=WS, wsb=1 << 30):
        return lib.raw_call("relattn_labeled_bwd", FAKE, FAKE, FAKE, aK, aV, ctypes.c_longlong(ths),
                            L, labels, ctypes.c_longlong(lbs), causal, ctypes.c_float(1.0), None,
                            1, 2, n, d, dtype, FAKE, G[0], G[1], G[2], daK, daV, ws,
                            ctypes.c_ulonglong(wsb), None)

    assert call(L=0) == 1
    assert call(L=257) == 1
    assert call(labels=None) == 1
    assert call(lbs=100) == 1                          # below n * n
    assert call(ths=8 * 64 - 1) == 1                   # below num_labels * d
    assert call(daK=None) == 1                         # a table without its gradient
    assert call(aV=TAB, daV=None) == 1
    assert call(causal=2) == 1
    assert call(ws=None) == 1
    assert call(wsb=16) == 1
    assert call(d=256, dtype=1) == 2
    nb = ctypes.c_ulonglong(0)
    assert lib.raw_call("relattn_labeled_bwd_workspace_size", 2, 3, 5, 8, ctypes.byref(nb)) == 0
    # per query row: m, 1/l, D and four values per label (R, Rv and the two bins)
    assert nb.value == 2 * 3 * 5 * (3 + 4 * 8) * 4
    assert lib.raw_call("relattn_labeled_bwd_workspace_size", 2, 3, 5, 0, ctypes.byref(nb)) == 1
