// Transformer-XL relative attention on the SIMT units ("Relative Position Encoding in
// Transformer-XL" page, the four-term score and the roles of u and v; "Relative position
// embeddings" page, section "Transformer-XL"):
//   A_ij = q_i.k_j + q_i.r_ij + u.k_j + v.r_ij = (q_i + u).k_j + (q_i + v).r_ij
//   z_i  = sum_j softmax_j(scale * A)_ij v_j
// r_ij = rel[h][(j - i) + n - 1], the projected encodings of every offset (a caller table).
// Terms (a) + (c) and (b) + (d) are each one dot product with the query row shifted by u or v
// (formed in fp32 from the inputs). One warp per query row; lane t computes both dot products
// of key j0 + t; fp32 arithmetic for bf16 and fp32 inputs, online softmax, P V on the lanes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "relattn_internal.h"

namespace relattn {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxD = 128;
constexpr int kPerLane = kMaxD / 32;

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float *x) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ static float one(const float *p) { return *p; }
    __device__ static void store(float *p, float x) { *p = x; }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float *x) {
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
__global__ void __launch_bounds__(kWarps * 32) txl_kernel(const TxlArgs a, int row_blocks) {
    __shared__ __align__(16) float s_qu[kWarps][kMaxD];
    __shared__ __align__(16) float s_qv[kWarps][kMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long bh = blockIdx.x / row_blocks;
    const int i = (int)(blockIdx.x % row_blocks) * kWarps + warp;
    if (i >= a.n) return;
    const int n = a.n, d = a.d;
    const int b = (int)(bh / a.H), h = (int)(bh % a.H);
    int valid = n;
    if (a.kv_len) valid = max(0, min(a.kv_len[b], n));
    const int jend = a.causal ? min(valid, i + 1) : valid;
    const T *q = static_cast<const T *>(a.q) + (bh * n + i) * d;
    const T *kb = static_cast<const T *>(a.k) + bh * (long long)n * d;
    const T *vbase = static_cast<const T *>(a.v) + bh * (long long)n * d;
    const T *rel = static_cast<const T *>(a.rel) + (long long)(a.shared ? 0 : h) * (2LL * n - 1) * d;
    const T *u = static_cast<const T *>(a.u) + (long long)(a.shared ? 0 : h) * d;
    const T *vb = static_cast<const T *>(a.vb) + (long long)(a.shared ? 0 : h) * d;
    float *qu = s_qu[warp], *qv = s_qv[warp];
    for (int c = lane; c < d; c += 32) {
        const float x = Vec<T>::one(q + c);
        qu[c] = (x + Vec<T>::one(u + c)) * a.scale;
        qv[c] = (x + Vec<T>::one(vb + c)) * a.scale;
    }
    __syncwarp();
    float acc[kPerLane];
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) acc[t] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int j0 = 0; j0 < jend; j0 += 32) {
        const int j = j0 + lane;
        const bool live = j < jend;
        float e = -INFINITY;
        if (live)
            e = dot_row<T>(qu, kb + (long long)j * d, d) +
                dot_row<T>(qv, rel + (long long)(j - i + n - 1) * d, d);
        const float m_new = fmaxf(m, warp_max(e));
        const float corr = expf(m - m_new);
        const float p = live ? expf(e - m_new) : 0.f;
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int t = 0; t < kPerLane; ++t) acc[t] *= corr;
        const int cnt = min(32, jend - j0);
        for (int t = 0; t < cnt; ++t) {
            const float pj = __shfl_sync(0xffffffffu, p, t);
            const T *vr = vbase + (long long)(j0 + t) * d;
#pragma unroll
            for (int uu = 0; uu < kPerLane; ++uu) {
                const int c = lane + 32 * uu;
                if (c < d) acc[uu] = fmaf(pj, Vec<T>::one(vr + c), acc[uu]);
            }
        }
        m = m_new;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *out = static_cast<T *>(a.out) + (bh * n + i) * d;
#pragma unroll
    for (int uu = 0; uu < kPerLane; ++uu) {
        const int c = lane + 32 * uu;
        if (c < d) Vec<T>::store(out + c, acc[uu] * inv);
    }
}

// The sinusoidal encodings of the relative offsets -(n-1) .. n-1: row o, components 2i and
// 2i + 1 = sin and cos of (o - (n - 1)) / 10000^(2i / d_model). The angle is formed in fp64
// (offsets of thousands times frequencies near 1 would lose digits in fp32), then rounded to
// the output type.
template <typename T>
__global__ void sinusoid_kernel(int n, int d_model, T *out) {
    const long long half = d_model / 2;
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (row, i) pair
    if (e >= (2LL * n - 1) * half) return;
    const long long row = e / half;
    const int i = (int)(e - row * half);
    const double pos = (double)(row - (n - 1));
    const double ang = pos * exp2(-(2.0 * i / d_model) * 13.287712379549449);  // log2(10000)
    T *o = out + row * d_model + 2 * i;
    Vec<T>::store(o, (float)sin(ang));
    Vec<T>::store(o + 1, (float)cos(ang));
}

}  // namespace

cudaError_t launch_sinusoid(int n, int d_model, int bf16, void *out, cudaStream_t s) {
    const long long pairs = (2LL * n - 1) * (d_model / 2);
    if (pairs <= 0) return cudaSuccess;
    const long long blocks = (pairs + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
    if (bf16)
        sinusoid_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(n, d_model, static_cast<__nv_bfloat16 *>(out));
    else
        sinusoid_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(n, d_model, static_cast<float *>(out));
    return cudaGetLastError();
}

cudaError_t launch_txl(const TxlArgs &a, cudaStream_t s) {
    if (a.d > kMaxD) return cudaErrorNotSupported;
    const int row_blocks = (a.n + kWarps - 1) / kWarps;
    const long long blocks = (long long)a.B * a.H * row_blocks;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
    if (a.bf16)
        txl_kernel<__nv_bfloat16><<<(unsigned)blocks, kWarps * 32, 0, s>>>(a, row_blocks);
    else
        txl_kernel<float><<<(unsigned)blocks, kWarps * 32, 0, s>>>(a, row_blocks);
    return cudaGetLastError();
}

}  // namespace relattn
