"""Exact index math of the oracle: clip labels and T5 buckets.

Pins: the page's statements (exact range, clamp, bucket count), and an integer closed form
that holds for the default constants (32 buckets, max_distance 128, bidirectional):
for a = |j - i| >= 8,
    8 + floor(ln(a/8) / ln(128/8) * 8) = 8 + floor(2 * log2(a/8)) = 2 + floor(log2(a^2)),
and floor(log2(x)) of a positive integer x is x.bit_length() - 1. This needs no logarithm,
so it checks the oracle's tie handling (a = 16, 32, 64 land exactly on integers).
"""
import json
import os

import pytest

import oracle
from oracle import t5

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _closed_form_default(delta):
    a = abs(delta)
    half = 16 if delta > 0 else 0
    if a < 8:
        return half + a
    return half + min(15, 2 + (a * a).bit_length() - 1)


def test_t5_default_matches_integer_closed_form():
    for dl in range(-4096, 4097):
        assert t5.t5_bucket(dl, 32, 128, True) == _closed_form_default(dl), dl


def test_t5_default_thresholds():
    # first |delta| of each log bucket 8..15 (lower half); from the closed form above
    firsts = {}
    for a in range(0, 300):
        b = t5.t5_bucket(-a, 32, 128, True)
        firsts.setdefault(b, a)
    assert [firsts[b] for b in range(8, 16)] == [8, 12, 16, 23, 32, 46, 64, 91]


def test_t5_page_statements():
    g = json.load(open(os.path.join(GOLDEN, "t5_page_facts.json")))
    B, D = g["num_buckets"], g["max_distance"]
    # exact for the first B/4 offsets when bidirectional (per sign half)
    for a in range(g["exact_bidirectional"]):
        assert t5.t5_bucket(-a, B, D, True) == a
        if a > 0:
            assert t5.t5_bucket(a, B, D, True) == B // 2 + a
    # exact for the first B/2 offsets when unidirectional; future keys share bucket 0
    for a in range(g["exact_unidirectional"]):
        assert t5.t5_bucket(-a, B, D, False) == a
    for dl in range(0, 500):
        assert t5.t5_bucket(dl, B, D, False) == 0
    # clamp to the last bucket of each half, for any distance
    assert t5.t5_bucket(-10 ** 9, B, D, True) == B // 2 - 1
    assert t5.t5_bucket(10 ** 9, B, D, True) == B - 1
    assert t5.t5_bucket(-10 ** 9, B, D, False) == B - 1
    # B x H table entries
    e = g["table_entries_t5_base"]
    assert e["B"] * e["H"] == e["entries"]


@pytest.mark.parametrize("nb,md,bidir", [(32, 128, True), (32, 128, False), (16, 40, True),
                                         (64, 1000, True), (8, 5, False), (4, 3, True)])
def test_t5_monotone_in_distance_and_in_range(nb, md, bidir):
    prev = -1
    for a in range(0, 3000):
        b = t5.t5_bucket(-a, nb, md, bidir)
        assert b >= prev
        assert 0 <= b < (nb // 2 if bidir else nb)
        prev = b
    if bidir:
        for a in range(1, 3000):
            assert t5.t5_bucket(a, nb, md, True) == nb // 2 + t5.t5_bucket(-a, nb, md, True)


def test_t5_log_steps_exact_at_powers():
    # at a = e*(D/e)**(m/c) with integer results the floor must not drop below m
    # default: e = 8, D/e = 16, c = 8 -> a = 8*2**(m/2): a = 16 (m=2), 32 (m=4), 64 (m=6)
    for a, m in [(16, 2), (32, 4), (64, 6), (128, 8)]:
        assert t5.log_steps(a, 8, 16, 128) == m
        assert t5.log_steps(a - 1, 8, 16, 128) == m - 1


def test_t5_rejects_degenerate_parameters():
    with pytest.raises(ValueError):
        t5.t5_bucket(3, 2, 128, True)     # exact range empty
    with pytest.raises(ValueError):
        t5.t5_bucket(3, 32, 8, True)      # max_distance not beyond the exact range


def test_label_matrices():
    lab = oracle.clip_labels(5, 7, 2)
    assert lab[0].tolist() == [2, 3, 4, 4, 4, 4, 4]
    assert lab[4].tolist() == [0, 0, 0, 1, 2, 3, 4]
    t = oracle.t5_labels(3, 3, 32, 128, True)
    assert t.tolist() == [[0, 17, 18], [1, 0, 17], [2, 1, 0]]
