// Device helpers shared by the kernels of librelattn.so (index math of the method).
#pragma once

#include <cstdint>

#include "relattn_internal.h"

namespace relattn {

// clip(x, k) = max(-k, min(k, x)) — paper summary, section 3.4 "Relative Position
// Representations: From Arbitrary Edges to Sequences".
__device__ __forceinline__ int clip_offset(int x, int k) { return max(-k, min(k, x)); }

// T5 bucket of the offset delta = j - i ("Relative position embeddings", section "T5"),
// with the exact thresholds computed on the host.
__device__ __forceinline__ int t5_bucket(int delta, const T5Buckets &t) {
    int offset = 0, a;
    if (t.bidir) {
        offset = delta > 0 ? t.half : 0;
        a = delta < 0 ? -delta : delta;
    } else {
        a = delta < 0 ? -delta : 0;
    }
    if (a < t.exact) return offset + a;
    int b = t.exact;
    for (int m = 0; m < t.nthr; ++m) b += (a >= t.thr[m]) ? 1 : 0;
    return offset + b;
}

// Scalar bias of offset delta = j - i for head h: a T5 bucket's table entry, ALiBi's
// -m_h |delta| ("Placement in the taxonomy": the T5 table replaced by a line), or the entry
// clip(delta, R) + R of a per-offset table (R the table's radius, hs its head stride).
__device__ __forceinline__ float scalar_bias(const float *bias, int kind, int H, int R,
                                             long long hs, const T5Buckets &t, int delta, int h) {
    if (kind == kBiasAlibi) return -bias[h] * (float)(delta < 0 ? -delta : delta);
    if (kind == kBiasTable) return bias[(long long)h * hs + clip_offset(delta, R) + R];
    return bias[(long long)t5_bucket(delta, t) * H + h];
}

}  // namespace relattn
