// Exact T5 bucket thresholds on the host.
//
// "Relative position embeddings" page, section "T5": a distance a below the exact range
// maps to itself; otherwise the bucket is
//     exact + floor( ln(a/exact) / ln(max_distance/exact) * (half - exact) ),
// clamped to the half's last bucket. The floor is of the exact real number, so the
// threshold of log step m (m = 1 .. half-1-exact) is the smallest integer a with
//     m <= c * ln(a/e) / ln(D/e)   <=>   D^m * e^c <= a^c * e^m      (c = half - exact).
// Both sides are products of integer powers; they are compared exactly with a small
// arbitrary-precision unsigned integer, never with a floating-point logarithm, so ties
// (a = 16, 32, 64 at the defaults) resolve the same way as the real-number formula.
#include <cstdint>
#include <vector>

#include "relattn_internal.h"

namespace relattn {
namespace {

struct Big {
    std::vector<uint32_t> limb{1};  // little-endian base 2^32, value 1

    void mul(uint32_t x) {
        uint64_t carry = 0;
        for (auto &l : limb) {
            const uint64_t t = (uint64_t)l * x + carry;
            l = (uint32_t)t;
            carry = t >> 32;
        }
        if (carry) limb.push_back((uint32_t)carry);
    }
    void mul_pow(uint32_t x, int e) {
        for (int i = 0; i < e; ++i) mul(x);
    }
    void trim() {
        while (limb.size() > 1 && limb.back() == 0) limb.pop_back();
    }
};

int cmp(Big a, Big b) {
    a.trim();
    b.trim();
    if (a.limb.size() != b.limb.size()) return a.limb.size() < b.limb.size() ? -1 : 1;
    for (size_t i = a.limb.size(); i-- > 0;)
        if (a.limb[i] != b.limb[i]) return a.limb[i] < b.limb[i] ? -1 : 1;
    return 0;
}

// true when log step m is reached at distance a: D^m * e^c <= a^c * e^m
bool reaches(uint32_t a, int m, uint32_t e, uint32_t D, int c) {
    Big lhs, rhs;
    lhs.mul_pow(D, m);
    lhs.mul_pow(e, c);
    rhs.mul_pow(a, c);
    rhs.mul_pow(e, m);
    return cmp(lhs, rhs) <= 0;
}

}  // namespace

bool t5_make_buckets(int num_buckets, int max_distance, int bidirectional, T5Buckets *b) {
    if (!b || num_buckets < 2 || num_buckets > 2 * kMaxT5Thresholds) return false;
    const int half = bidirectional ? num_buckets / 2 : num_buckets;
    const int exact = half / 2;
    if (exact < 1 || max_distance <= exact) return false;
    const int c = half - exact;
    b->half = half;
    b->exact = exact;
    b->bidir = bidirectional ? 1 : 0;
    b->nthr = half - 1 - exact;
    if (b->nthr > kMaxT5Thresholds) return false;
    for (int m = 1; m <= b->nthr; ++m) {
        // a = max_distance always reaches step m <= c; binary search the first a >= exact
        uint32_t lo = (uint32_t)exact, hi = (uint32_t)max_distance;
        while (lo < hi) {
            const uint32_t mid = lo + (hi - lo) / 2;
            if (reaches(mid, m, (uint32_t)exact, (uint32_t)max_distance, c))
                hi = mid;
            else
                lo = mid + 1;
        }
        b->thr[m - 1] = (int)lo;
    }
    b->sat = b->nthr > 0 ? b->thr[b->nthr - 1] : exact;
    return true;
}

}  // namespace relattn
