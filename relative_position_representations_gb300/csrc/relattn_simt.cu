// fp32 SIMT path (no tensor cores) and the label kernel.
//
// fp32 keeps the whole computation in IEEE fp32 with accurate expf (this file is built
// without fast-math), one warp per query row: lanes split the head dimension d, a warp
// reduction forms each logit, and an online softmax accumulates the output. TF32 tensor
// cores would not meet a 1e-5 relative bound, so this path stays on the FMA pipes.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "relattn_internal.h"

namespace relattn {
namespace {

constexpr int kWarpsPerBlock = 4;
constexpr int kMaxPerLane = 4;  // d <= 128

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Shaw ("Self-Attention with Relative Position Representations" page, section 3.4, eqs. 3
// and 4) or a scalar offset bias ("Relative position embeddings", sections "T5" and
// "Placement in the taxonomy") forward for one query row per warp.
template <bool T5>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    simt_f32_kernel(const SimtArgs a, const T5Buckets t5) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarpsPerBlock + warp;
    const long long rows = (long long)a.B * a.H * a.n;
    if (row >= rows) return;
    const int n = a.n, d = a.d;
    const long long bh = row / n;
    const int i = (int)(row % n);
    const int b = (int)(bh / a.H), h = (int)(bh % a.H);
    int valid = n;
    if (a.kv_len) valid = max(0, min(a.kv_len[b], n));
    const int jend = a.causal ? min(valid, i + 1) : valid;

    float qv[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
        const int c = lane + 32 * t;
        qv[t] = c < d ? a.q[row * d + c] : 0.f;
        acc[t] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float *kb = a.k + bh * (long long)n * d;
    const float *vb = a.v + bh * (long long)n * d;
    const float *tk = (!T5 && a.aK) ? a.aK + (long long)h * a.ths : nullptr;
    const float *tv = (!T5 && a.aV) ? a.aV + (long long)h * a.ths : nullptr;
    for (int j = 0; j < jend; ++j) {
        int r = 0;
        if (!T5) r = clip_offset(j - i, a.clip_k) + a.clip_k;
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxPerLane; ++t) {
            const int c = lane + 32 * t;
            if (c < d) {
                float kk = kb[(long long)j * d + c];
                if (tk) kk += tk[(long long)r * d + c];
                part = fmaf(qv[t], kk, part);
            }
        }
        float e = warp_sum(part) * a.scale;
        if (T5) e += scalar_bias(a.bias, a.bias_kind, a.H, a.bias_R, a.bias_hs, t5, j - i, h);
        const float m_new = fmaxf(m, e);
        const float corr = expf(m - m_new);  // m = -inf on the first key -> 0
        const float p = expf(e - m_new);
        l = l * corr + p;
#pragma unroll
        for (int t = 0; t < kMaxPerLane; ++t) {
            const int c = lane + 32 * t;
            if (c < d) {
                float vv = vb[(long long)j * d + c];
                if (tv) vv += tv[(long long)r * d + c];
                acc[t] = fmaf(p, vv, acc[t] * corr);
            }
        }
        m = m_new;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
        const int c = lane + 32 * t;
        if (c < d) a.out[row * d + c] = acc[t] * inv;
    }
}

// Edge label of every (i, j): clip row (kind 0) or T5 bucket (kind 1).
__global__ void labels_kernel(int kind, int clip_k, const T5Buckets t5, int n_q, int n_k,
                              int *labels) {
    const long long total = (long long)n_q * n_k;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(idx / n_k), j = (int)(idx % n_k);
        labels[idx] = kind == 0 ? clip_offset(j - i, clip_k) + clip_k : t5_bucket(j - i, t5);
    }
}

}  // namespace

cudaError_t launch_simt_f32(const SimtArgs &a, const T5Buckets *t5, cudaStream_t s) {
    const long long rows = (long long)a.B * a.H * a.n;
    if (rows == 0) return cudaSuccess;
    const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (t5) {
        simt_f32_kernel<true><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, s>>>(a, *t5);
    } else {
        T5Buckets none{};
        simt_f32_kernel<false><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, s>>>(a, none);
    }
    return cudaGetLastError();
}

cudaError_t launch_labels(int kind, int clip_k, const T5Buckets *t5, int n_q, int n_k,
                          int *labels, cudaStream_t s) {
    const long long total = (long long)n_q * n_k;
    if (total == 0) return cudaSuccess;
    T5Buckets none{};
    const long long want = (total + 255) / 256;
    const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
    labels_kernel<<<blocks, 256, 0, s>>>(kind, clip_k, t5 ? *t5 : none, n_q, n_k, labels);
    return cudaGetLastError();
}

}  // namespace relattn
