"""Exact T5 relative-position bucketing (oracle side).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference leg, never by the product path.

Source: "Relative position embeddings" page, section "T5": the logit gets a scalar
b^(h)[beta(j - i)], with B buckets (default 32) and max_distance (default 128). The page
says the bucketing is exact for the first B/2 offsets (B/4 when bidirectional) and
logarithmic after that,

    beta(a) = a                                                     if a < B_exact
    beta(a) = B_exact + floor( ln(a / B_exact) / ln(D_max / B_exact) * (B - B_exact) )
                                                                    otherwise,
    clamped to B - 1.

Readings taken where the page is garbled or silent:
  * bidirectional: the B buckets split into two halves of B/2, one per sign; inside a
    half B_exact = (B/2)/2 and the formula uses the half's size B/2 in place of B.
    Offsets j - i > 0 use the upper half (bucket + B/2), offsets <= 0 the lower half.
  * unidirectional: one half of size B, B_exact = B/2, a = max(i - j, 0), so keys after
    the query all land in bucket 0.
  * the floor is taken of the exact real number: ties such as a = 16, 32, 64 at the
    default constants (where the real value is an integer) resolve upward, with no
    floating-point rounding involved. This is done with integer arithmetic:
        m <= c * ln(a/e) / ln(D/e)  <=>  D**m * e**c <= a**c * e**m     (c = half - e)
"""
from __future__ import annotations

import math


def _halves(num_buckets: int, bidirectional: bool) -> tuple[int, int]:
    half = num_buckets // 2 if bidirectional else num_buckets
    exact = half // 2
    return half, exact


def log_steps(a: int, exact: int, half: int, max_distance: int) -> int:
    """Largest integer m >= 0 with m <= (half-exact) * ln(a/exact) / ln(max_distance/exact).

    Requires a >= exact >= 1 and max_distance > exact. Exact integer arithmetic.
    """
    c = half - exact
    D, e = max_distance, exact

    def holds(m: int) -> bool:
        return D ** m * e ** c <= a ** c * e ** m

    guess = int(math.floor(c * math.log(a / e) / math.log(D / e)))
    m = max(guess, 0)
    while m > 0 and not holds(m):
        m -= 1
    while holds(m + 1):
        m += 1
    return m


def t5_bucket(delta: int, num_buckets: int = 32, max_distance: int = 128,
              bidirectional: bool = True) -> int:
    """Bucket index of the relative offset delta = j - i (exact)."""
    half, exact = _halves(num_buckets, bidirectional)
    if exact < 1:
        raise ValueError("num_buckets too small: the exact range would be empty")
    if max_distance <= exact:
        raise ValueError("max_distance must exceed the exact range")
    if bidirectional:
        offset = half if delta > 0 else 0
        a = abs(delta)
    else:
        offset = 0
        a = max(-delta, 0)
    if a < exact:
        return offset + a
    m = log_steps(a, exact, half, max_distance)
    return offset + min(exact + m, half - 1)


def bucket_of_offset_table(n: int, num_buckets: int, max_distance: int,
                           bidirectional: bool) -> list[int]:
    """Bucket for every offset j - i in [-(n-1), n-1]; index (j - i) + (n - 1)."""
    return [t5_bucket(dl, num_buckets, max_distance, bidirectional)
            for dl in range(-(n - 1), n)]
