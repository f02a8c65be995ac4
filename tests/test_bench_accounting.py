"""The bench's algorithmic FLOP and byte counts (the roofline numerators), checked on CPU.

The per-workload figures are worked out by hand from the counting rule (4*d per unmasked
(query, key) pair for Q.K^T and P.V, 2*d*n per reachable table row and table term, bytes of
Q, O, the K and V rows below kv_len and each table once) and compared with bench.py; the
per-row counts used for the CPU baseline must add up to the whole-launch count.
"""
import numpy as np
import pytest

import bench
from relative_position_representations_gb300 import workloads as wl


def test_pairs_per_sequence():
    w = wl.Workload("t", B=1, H=1, n=4, d=8, dtype="f32", causal=True)
    assert bench.pairs_per_sequence(w, None) == 10          # 1 + 2 + 3 + 4
    assert bench.pairs_per_sequence(w, 2) == 7              # 1 + 2 + 2 + 2
    assert bench.pairs_per_sequence(w.replace(causal=False), 3) == 12
    assert bench.pairs_per_sequence(w.replace(causal=False), 0) == 0


def test_big_decoder_counts():
    w = wl.WORKLOADS["big_decoder"]   # B32 H16 n256 d64 k16 causal, both tables
    BH = 32 * 16
    flops = 4 * 64 * (256 * 257 // 2) * BH + 2 * 64 * 256 * 17 * 2 * BH
    assert bench.algorithmic_flops(w, None) == pytest.approx(flops, rel=1e-12)
    assert flops == pytest.approx(4.88e9, rel=2e-3)
    byts = 2 * (4 * BH * 256 * 64) + 2 * 16 * 33 * 64 * 2
    assert bench.algorithmic_bytes(w, None) == pytest.approx(byts, rel=1e-12)


def test_long_keyonly_and_t5_counts():
    w = wl.WORKLOADS["long_keyonly"]  # B4 H16 n4096 d128 k64 causal, key table only
    BH = 64
    flops = 4 * 128 * (4096 * 4097 // 2) * BH + 2 * 128 * 4096 * 65 * 1 * BH
    assert bench.algorithmic_flops(w, None) == pytest.approx(flops, rel=1e-12)
    assert flops == pytest.approx(279.3e9, rel=1e-3)
    t5 = wl.WORKLOADS["t5_bias"]      # B8 H12 n2048 d64, bidirectional
    assert bench.algorithmic_flops(t5, None) == pytest.approx(4 * 64 * 2048 * 2048 * 96, rel=1e-12)
    assert bench.algorithmic_bytes(t5, None) == pytest.approx(
        2 * 4 * 96 * 2048 * 64 + 4 * 32 * 12, rel=1e-12)


def test_base_encoder_counts_follow_the_key_lengths():
    w = wl.WORKLOADS["base_encoder"]  # B64 H8 n128 d64 k16, bidirectional, padded keys
    kv = [32 + (b * 7) % 97 for b in range(64)]
    pairs = sum(128 * x for x in kv) * 8
    flops = 4 * 64 * pairs + 2 * 64 * 128 * 33 * 2 * 64 * 8
    assert bench.algorithmic_flops(w, kv) == pytest.approx(flops, rel=1e-12)
    byts = 2 * (2 * 64 * 8 * 128 * 64 + 2 * sum(kv) * 8 * 64) + 2 * 8 * 33 * 64 * 2
    assert bench.algorithmic_bytes(w, kv) == pytest.approx(byts, rel=1e-12)
    # no padding: the unpadded figure of the configuration table
    assert bench.algorithmic_flops(w, None) == pytest.approx(2.70e9, rel=2e-3)


def test_decode_counts():
    w = wl.Workload("dec", B=2, H=3, n=100, d=64, dtype="bf16", kind="decode", clip_k=4,
                    causal=True)
    cl = [10, 0]
    flops = 4 * 64 * 10 * 3 + 2 * 64 * 5 * 2 * 3      # the empty cache adds nothing
    assert bench.algorithmic_flops(w, cl) == pytest.approx(flops, rel=1e-12)
    byts = 2 * (2 * 2 * 3 * 64 + 2 * 10 * 3 * 64 + 3 * 5 * 64 * 2) + 4 * 2
    assert bench.algorithmic_bytes(w, cl) == pytest.approx(byts, rel=1e-12)


def test_scalar_bias_and_labelled_counts():
    alibi = wl.Workload("a", B=2, H=3, n=10, d=16, dtype="bf16", kind="alibi", causal=True)
    assert bench.algorithmic_flops(alibi, None) == pytest.approx(4 * 16 * 55 * 6, rel=1e-12)
    assert bench.algorithmic_bytes(alibi, None) == pytest.approx(2 * 4 * 6 * 10 * 16 + 4 * 3)
    off = alibi.replace(kind="offset", clip_k=5, causal=False, shared_tables=True)
    assert bench.algorithmic_bytes(off, None) == pytest.approx(2 * 4 * 6 * 10 * 16 + 4 * 11)
    lab = wl.Workload("l", B=2, H=3, n=10, d=16, dtype="bf16", kind="labeled", num_labels=7)
    flops = 4 * 16 * 100 * 6 + 2 * 16 * 10 * 7 * 2 * 6
    assert bench.algorithmic_flops(lab, None) == pytest.approx(flops, rel=1e-12)
    byts = 2 * 4 * 6 * 10 * 16 + 2 * 3 * 7 * 16 * 2 + 2 * 10 * 10
    assert bench.algorithmic_bytes(lab, None) == pytest.approx(byts, rel=1e-12)


@pytest.mark.parametrize("name", ["base_encoder", "big_decoder"])
def test_row_counts_add_up_to_the_launch(name):
    w = wl.WORKLOADS[name].replace(B=3)
    kv = [40, 128, 77] if w.kv_len_range else None
    rows = np.arange(w.B * w.H * w.n)
    assert bench.row_flops(w, kv, rows) == pytest.approx(bench.algorithmic_flops(w, kv), rel=1e-12)


def test_labelled_row_counts_add_up_to_the_launch():
    w = wl.Workload("l", B=2, H=2, n=9, d=8, dtype="f32", kind="labeled", num_labels=5,
                    causal=True)
    rows = np.arange(w.B * w.H * w.n)
    assert bench.row_flops(w, [9, 4], rows) == pytest.approx(bench.algorithmic_flops(w, [9, 4]))


def test_txl_counts_three_dot_products_per_pair_and_the_offset_table():
    # B=1, H=1, n=3, d=2, causal: pairs 1 + 2 + 3 = 6; FLOPs 6 d per pair = 72. Bytes (bf16):
    # q, out 2 * 6 elements, k, v 2 * 6, rel (2n - 1) * d = 10 and u, v 2 * d = 4 -> 38 * 2
    w = wl.Workload("x", B=1, H=1, n=3, d=2, dtype="bf16", kind="txl", causal=True)
    assert bench.algorithmic_flops(w, None) == 72.0
    assert bench.algorithmic_bytes(w, None) == 76.0
