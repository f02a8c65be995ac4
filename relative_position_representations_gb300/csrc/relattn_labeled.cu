// Relation-aware attention over arbitrary labelled edges ("Self-Attention with Relative
// Position Representations" page, section "Relation-Aware Self-Attention: The Core
// Modification": every edge (i, j) of the input graph carries its own a^K_ij, a^V_ij; here
// they are rows of two tables picked by a label matrix, the general form that section 3.4
// specialises to clip(j - i, k) + k):
//
//   e_ij = scale * q_i . (k_j + w^K[L_b[i, j]])         (eq. 4)
//   z_i  = sum_j softmax_j(e)_ij * (v_j + w^V[L_b[i, j]]) (eq. 3)
//
// computed in the split form of "Efficient Implementation": R_ir = scale * q_i . w^K_r once
// per row and a gather R_i[L_ij] per edge; the value term through the bins
// beta_ir = sum over {j : L_ij = r} of p_ij, then z_i += beta_i . W^V. Nothing of size
// n x n x d is formed.
//
// SIMT, fp32 arithmetic (bf16 or fp32 inputs), one warp per query row: lane t computes the
// logit of key j0 + t of each 32-key chunk (its whole dot product), the warp keeps an online
// softmax, and the lanes split the head dimension for P . V. With no structure in the labels
// there is no band to exploit: every edge takes a shared-memory gather (and a shared-memory
// add into its bin).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "relattn_internal.h"

namespace relattn {
namespace {

constexpr int kWarps = 8;        // query rows per CTA
constexpr int kMaxD = 128;
constexpr int kPerLane = kMaxD / 32;

template <typename T>
struct Vec;

template <>
struct Vec<float> {
    static constexpr int N = 4;  // elements per 16-byte load
    __device__ static void load(const float *p, float *x) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    }
    __device__ static float one(const float *p) { return *p; }
    __device__ static void store(float *p, float x) { *p = x; }
};

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float *x) {
        // a bf16 value is the upper 16 bits of the fp32 value it stands for
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            x[2 * t] = __uint_as_float(w[t] << 16);
            x[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
        }
    }
    __device__ static float one(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ static void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// dot product of the scaled query row in shared memory with a d-element row in global memory
template <typename T>
__device__ __forceinline__ float dot_row(const float *sq, const T *row, int d) {
    constexpr int N = Vec<T>::N;
    float acc = 0.f;
    for (int c = 0; c < d; c += N) {
        float x[N];
        Vec<T>::load(row + c, x);
#pragma unroll
        for (int t = 0; t < N; ++t) acc = fmaf(sq[c + t], x[t], acc);
    }
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) labeled_kernel(const LabeledArgs a, int row_blocks) {
    __shared__ __align__(16) float s_q[kWarps][kMaxD];
    __shared__ float s_r[kWarps][kMaxLabels];
    __shared__ float s_beta[kWarps][kMaxLabels];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long bh = blockIdx.x / row_blocks;
    const int i = (int)(blockIdx.x % row_blocks) * kWarps + warp;
    if (i >= a.n) return;  // whole warps leave; nothing below synchronises the block
    const int n = a.n, d = a.d, L = a.num_labels;
    const int b = (int)(bh / a.H), h = (int)(bh % a.H);
    int valid = n;
    if (a.kv_len) valid = max(0, min(a.kv_len[b], n));
    const int jend = a.causal ? min(valid, i + 1) : valid;

    const T *q = static_cast<const T *>(a.q);
    const T *kb = static_cast<const T *>(a.k) + bh * (long long)n * d;
    const T *vb = static_cast<const T *>(a.v) + bh * (long long)n * d;
    const T *tk = a.aK ? static_cast<const T *>(a.aK) + (long long)h * a.ths : nullptr;
    const T *tv = a.aV ? static_cast<const T *>(a.aV) + (long long)h * a.ths : nullptr;
    const bool labelled = tk != nullptr || tv != nullptr;
    const uint8_t *lrow = labelled ? a.labels + (long long)b * a.lbs + (long long)i * n : nullptr;
    float *sq = s_q[warp];
    float *R = s_r[warp];
    float *beta = s_beta[warp];

    // the scaled query row, then R_r = scale * q . w^K_r (one lane per table row)
    for (int c = lane; c < d; c += 32) sq[c] = Vec<T>::one(q + (bh * n + i) * d + c) * a.scale;
    __syncwarp();
    for (int r = lane; r < L && labelled; r += 32) {
        if (tk) R[r] = dot_row<T>(sq, tk + (long long)r * d, d);
        if (tv) beta[r] = 0.f;
    }
    __syncwarp();

    float acc[kPerLane];
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) acc[u] = 0.f;
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    for (int j0 = 0; j0 < jend; j0 += 32) {
        const int j = j0 + lane;
        const bool live = j < jend;
        int lab = 0;
        float e = -INFINITY;
        if (live) {
            if (labelled) {
                lab = lrow[j];
                if (lab >= L) {  // no table row: recorded, and read as the last row
                    bad = true;
                    lab = L - 1;
                }
            }
            e = dot_row<T>(sq, kb + (long long)j * d, d);
            if (tk) e += R[lab];
        }
        const float m_new = fmaxf(m, warp_max(e));  // finite: key j0 is live
        const float corr = expf(m - m_new);         // 0 on the first chunk
        const float p = live ? expf(e - m_new) : 0.f;
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int u = 0; u < kPerLane; ++u) acc[u] *= corr;
        if (tv) {
            if (corr != 1.f)
                for (int r = lane; r < L; r += 32) beta[r] *= corr;
            __syncwarp();
            if (live) atomicAdd(&beta[lab], p);
            __syncwarp();
        }
        const int cnt = min(32, jend - j0);
        for (int t = 0; t < cnt; ++t) {
            const float pj = __shfl_sync(0xffffffffu, p, t);
            const T *vr = vb + (long long)(j0 + t) * d;
#pragma unroll
            for (int u = 0; u < kPerLane; ++u) {
                const int c = lane + 32 * u;
                if (c < d) acc[u] = fmaf(pj, Vec<T>::one(vr + c), acc[u]);
            }
        }
        m = m_new;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && a.err)
        atomicCAS(a.err, 0, (int)kLabelOutOfRange);
    __syncwarp();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *out = static_cast<T *>(a.out) + (bh * n + i) * d;
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) {
        const int c = lane + 32 * u;
        if (c >= d) continue;
        float z = acc[u];
        if (tv)
            for (int r = 0; r < L; ++r) z = fmaf(beta[r], Vec<T>::one(tv + (long long)r * d + c), z);
        Vec<T>::store(out + c, z * inv);
    }
}

}  // namespace

cudaError_t launch_labeled(const LabeledArgs &a, cudaStream_t s) {
    if (a.d > kMaxD || a.num_labels > kMaxLabels) return cudaErrorNotSupported;
    const long long bh = (long long)a.B * a.H;
    const int row_blocks = (a.n + kWarps - 1) / kWarps;
    const long long blocks = bh * row_blocks;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
    if (a.bf16)
        labeled_kernel<__nv_bfloat16><<<(unsigned)blocks, kWarps * 32, 0, s>>>(a, row_blocks);
    else
        labeled_kernel<float><<<(unsigned)blocks, kWarps * 32, 0, s>>>(a, row_blocks);
    return cudaGetLastError();
}

}  // namespace relattn
