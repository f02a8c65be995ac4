// Gradients of the scalar offset-bias forwards: the T5 bucketed bias ("Relative position
// embeddings" page, section "T5"), ALiBi's -m_h |j - i| and a learned scalar per offset
// clipped at a radius (same page, "Placement in the taxonomy").
//
// The pages give only the forward pass; the gradients are the chain rule through it. With
// e_ij = scale q_i . k_j + b_h(j - i), p = softmax_j(e), dp_ij = dz_i . v_j,
// de_ij = p_ij (dp_ij - D_i), D_i = sum_j p_ij dp_ij:
//   dq_i = scale sum_j de_ij k_j,  dk_j = scale sum_i de_ij q_i,  dv_j = sum_i p_ij dz_i,
// and the bias enters only through the offset, so every parameter gradient is a sum of
//   G_h(o) = sum over (b, i) of de_{i, i+o},   o = -(n-1) .. n-1:
//   T5:    dbias[bucket, h] = sum over offsets o of that bucket of G_h(o)
//   ALiBi: dm_h = -sum_o |o| G_h(o)                 (d e_ij / d m_h = -|j - i|)
//   table: dtable[h, r] = sum over o with clip(o, R) + R = r of G_h(o) (a shared row sums
//          over the heads).
//
// Three kernels, fp32 arithmetic on the SIMT units (inputs bf16 or fp32). The bias is a
// scalar per offset, so no step is a dense contraction beyond the two per-key dot products.
//   rows  one warp per query row (8 rows of one head per CTA): the head's bias over every
//         offset in shared memory, one pass for m, l and D (online), a second for dq and
//         de, whose per-offset sums collect in shared memory and go to G with one atomic
//         add per offset and CTA; per row m, 1/l and D go to the workspace.
//   keys  one warp per key: dk and dv over the rows that see it, from the per-row values.
//   param one CTA per head (or per table row set): G to the parameter's gradient.
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "relattn_internal.h"

namespace relattn {
namespace bbwd {

constexpr int kWarps = 8;    // rows or keys per CTA
constexpr int kMaxPer = 4;   // d <= 128: elements per lane
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ float ld(const float *p, long long i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, long long i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
struct Params {
    const T *q, *k, *v, *dz;
    const float *bias;
    int kind, R;        // BiasKind; table radius
    int nbk;            // T5: number of buckets
    long long hs;       // table: elements between heads' rows (0 = one shared row)
    T5Buckets t5;
    int causal;
    float scale;
    const int *kv_len;
    int B, H, n, d;
    float *dq, *dk, *dv, *dbias;
    float *rec;  // per row: m, 1/l, D
    float *G;    // [H, 2n - 1]: sum of de per offset (index o + n - 1)
};

__device__ __forceinline__ int keys_of(const int *kv_len, int b, int n) {
    return kv_len ? max(0, min(kv_len[b], n)) : n;
}

// the head's bias of every offset, index o + n - 1
template <typename T>
__device__ __forceinline__ void bias_row(const Params<T> &p, int h, float *bo) {
    const int nb = 2 * p.n - 1;
    for (int o = threadIdx.x; o < nb; o += kThreads)
        bo[o] = scalar_bias(p.bias, p.kind, p.H, p.R, p.hs, p.t5, o - (p.n - 1), h);
}

// ---------------------------------------------------------------------------------- rows
template <typename T>
__global__ void __launch_bounds__(kThreads) bias_bwd_rows(const Params<T> p) {
    extern __shared__ float sm[];
    const int n = p.n, nb = 2 * n - 1, d = p.d;
    float *bo = sm, *gs = sm + nb;  // bias and the CTA's de sums, both over the offsets
    const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    bias_row(p, h, bo);
    for (int o = threadIdx.x; o < nb; o += kThreads) gs[o] = 0.f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kWarps + warp;
    if (i < n) {  // (no early return: every thread reaches the flush below)
        const long long row = (long long)bh * n + i;
        const int nk = keys_of(p.kv_len, b, n);
        const int jend = p.causal ? min(nk, i + 1) : nk;  // keys 0 .. jend-1 are allowed
        const float *bi = bo + (n - 1 - i);                 // bias of key j: bi[j]
        float qv[kMaxPer], gv[kMaxPer], acc[kMaxPer];
#pragma unroll
        for (int t = 0; t < kMaxPer; ++t) {
            const int c = lane + 32 * t;
            qv[t] = c < d ? ld(p.q, row * d + c) : 0.f;
            gv[t] = c < d ? ld(p.dz, row * d + c) : 0.f;
            acc[t] = 0.f;
        }
        const long long kv0 = (long long)bh * n;  // first key row of this head
        // ---- pass 1: m, l and D = sum p dp (every lane holds the same values)
        float m = -INFINITY, l = 0.f, S = 0.f;  // S = sum exp(e - m) dp
        for (int j = 0; j < jend; ++j) {
            float s = 0.f, sv = 0.f;
#pragma unroll
            for (int t = 0; t < kMaxPer; ++t) {
                const int c = lane + 32 * t;
                if (c < d) {
                    s = fmaf(qv[t], ld(p.k, (kv0 + j) * d + c), s);
                    sv = fmaf(gv[t], ld(p.v, (kv0 + j) * d + c), sv);
                }
            }
            s = warp_sum(s);
            sv = warp_sum(sv);
            const float e = p.scale * s + bi[j];
            if (e > m) {
                const float a = __expf(m - e);  // 0 when m = -inf
                l *= a;
                S *= a;
                m = e;
            }
            const float pe = __expf(e - m);
            l += pe;
            S = fmaf(pe, sv, S);
        }
        const float D = l > 0.f ? S / l : 0.f;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        // ---- pass 2: dq and the per-offset sums of de
        for (int j = 0; j < jend; ++j) {
            float s = 0.f, sv = 0.f, kv[kMaxPer];
#pragma unroll
            for (int t = 0; t < kMaxPer; ++t) {
                const int c = lane + 32 * t;
                kv[t] = c < d ? ld(p.k, (kv0 + j) * d + c) : 0.f;
                s = fmaf(qv[t], kv[t], s);
                if (c < d) sv = fmaf(gv[t], ld(p.v, (kv0 + j) * d + c), sv);
            }
            s = warp_sum(s);
            sv = warp_sum(sv);
            const float pr = __expf(p.scale * s + bi[j] - m) * inv_l;
            const float de = pr * (sv - D);
#pragma unroll
            for (int t = 0; t < kMaxPer; ++t) acc[t] = fmaf(p.scale * de, kv[t], acc[t]);
            if (lane == 0) atomicAdd(gs + (j - i + n - 1), de);
        }
#pragma unroll
        for (int t = 0; t < kMaxPer; ++t) {
            const int c = lane + 32 * t;
            if (c < d) p.dq[row * d + c] = acc[t];
        }
        if (lane == 0) {
            float *rec = p.rec + row * 3;
            rec[0] = m;
            rec[1] = inv_l;
            rec[2] = D;
        }
    }
    __syncthreads();
    float *G = p.G + (long long)h * nb;
    for (int o = threadIdx.x; o < nb; o += kThreads) {
        const float g = gs[o];
        if (g != 0.f) atomicAdd(G + o, g);
    }
}

// ---------------------------------------------------------------------------------- keys
template <typename T>
__global__ void __launch_bounds__(kThreads) bias_bwd_keys(const Params<T> p) {
    extern __shared__ float bo[];  // the head's bias over the offsets
    const int n = p.n, d = p.d;
    const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
    bias_row(p, h, bo);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * kWarps + warp;
    if (j >= n) return;  // (no barrier follows)
    const long long key = (long long)bh * n + j;
    const int nk = keys_of(p.kv_len, b, n);
    float kv[kMaxPer], vv[kMaxPer], dk[kMaxPer], dv[kMaxPer];
#pragma unroll
    for (int t = 0; t < kMaxPer; ++t) {
        const int c = lane + 32 * t;
        kv[t] = c < d ? ld(p.k, key * d + c) : 0.f;
        vv[t] = c < d ? ld(p.v, key * d + c) : 0.f;
        dk[t] = 0.f;
        dv[t] = 0.f;
    }
    if (j < nk) {  // a padded key gets no gradient
        const long long q0 = (long long)bh * n;
        for (int i = p.causal ? j : 0; i < n; ++i) {
            float s = 0.f, sv = 0.f, qv[kMaxPer], gv[kMaxPer];
#pragma unroll
            for (int t = 0; t < kMaxPer; ++t) {
                const int c = lane + 32 * t;
                qv[t] = c < d ? ld(p.q, (q0 + i) * d + c) : 0.f;
                gv[t] = c < d ? ld(p.dz, (q0 + i) * d + c) : 0.f;
                s = fmaf(qv[t], kv[t], s);
                sv = fmaf(gv[t], vv[t], sv);
            }
            s = warp_sum(s);
            sv = warp_sum(sv);
            const float *rec = p.rec + (q0 + i) * 3;
            const float pr = __expf(p.scale * s + bo[j - i + n - 1] - rec[0]) * rec[1];
            const float de = pr * (sv - rec[2]);
#pragma unroll
            for (int t = 0; t < kMaxPer; ++t) {
                dk[t] = fmaf(p.scale * de, qv[t], dk[t]);
                dv[t] = fmaf(pr, gv[t], dv[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kMaxPer; ++t) {
        const int c = lane + 32 * t;
        if (c < d) {
            p.dk[key * d + c] = dk[t];
            p.dv[key * d + c] = dv[t];
        }
    }
}

// ---------------------------------------------------------------------------------- param
// T5 and ALiBi: one CTA per head. Table: one CTA per table row set (per head, or one for a
// shared row, summing over every head). Every entry of the gradient is written.
template <typename T>
__global__ void __launch_bounds__(kThreads) bias_bwd_param(const Params<T> p) {
    extern __shared__ float acc[];  // T5: per bucket; table: per reachable table row
    __shared__ float red[kWarps];
    const int n = p.n, nb = 2 * n - 1;
    const int tid = threadIdx.x;
    if (p.kind == kBiasAlibi) {
        const int h = blockIdx.x;
        const float *G = p.G + (long long)h * nb;
        float s = 0.f;
        for (int o = tid; o < nb; o += kThreads) s = fmaf((float)abs(o - (n - 1)), G[o], s);
        s = warp_sum(s);
        if ((tid & 31) == 0) red[tid >> 5] = s;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < kWarps; ++w) t += red[w];
            p.dbias[h] = -t;
        }
        return;
    }
    if (p.kind == kBiasBuckets) {
        const int h = blockIdx.x, nbk = p.nbk;
        for (int c = tid; c < nbk; c += kThreads) acc[c] = 0.f;
        __syncthreads();
        const float *G = p.G + (long long)h * nb;
        for (int o = tid; o < nb; o += kThreads) {
            const float g = G[o];
            if (g != 0.f) atomicAdd(acc + t5_bucket(o - (n - 1), p.t5), g);
        }
        __syncthreads();
        for (int c = tid; c < nbk; c += kThreads) p.dbias[(long long)c * p.H + h] = acc[c];
        return;
    }
    // table: rows r = clip(o, R) + R; offsets reach rows lo .. hi only
    const int R = p.R;
    const int lo = max(0, R - (n - 1)), hi = min(2 * R, R + (n - 1));
    for (int c = tid; c <= hi - lo; c += kThreads) acc[c] = 0.f;
    __syncthreads();
    const int h0 = p.hs == 0 ? 0 : (int)blockIdx.x, h1 = p.hs == 0 ? p.H : h0 + 1;
    for (int h = h0; h < h1; ++h) {
        const float *G = p.G + (long long)h * nb;
        for (int o = tid; o < nb; o += kThreads) {
            const float g = G[o];
            if (g != 0.f) atomicAdd(acc + (clip_offset(o - (n - 1), R) + R - lo), g);
        }
    }
    __syncthreads();
    float *dt = p.dbias + (long long)blockIdx.x * p.hs;
    for (long long r = tid; r <= 2LL * R; r += kThreads)
        dt[r] = (r >= lo && r <= hi) ? acc[r - lo] : 0.f;
}

template <typename T>
cudaError_t launch_t(const BiasBwdArgs &a, const T5Buckets *t5, cudaStream_t s) {
    Params<T> p;
    p.q = static_cast<const T *>(a.q);
    p.k = static_cast<const T *>(a.k);
    p.v = static_cast<const T *>(a.v);
    p.dz = static_cast<const T *>(a.dout);
    p.bias = a.bias;
    p.kind = a.kind;
    p.R = a.radius;
    p.nbk = a.num_buckets;
    p.hs = a.head_stride;
    p.t5 = t5 ? *t5 : T5Buckets{};
    p.causal = a.causal;
    p.scale = a.scale;
    p.kv_len = a.kv_len;
    p.B = a.B;
    p.H = a.H;
    p.n = a.n;
    p.d = a.d;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.dbias = a.dbias;
    const long long nb = 2LL * a.n - 1;
    p.rec = static_cast<float *>(a.workspace);
    p.G = p.rec + bias_bwd_rec_floats(a.B, a.H, a.n);
    const size_t rows_smem = (size_t)2 * nb * sizeof(float), keys_smem = (size_t)nb * sizeof(float);
    {  // shared memory above the default 48 KB: opt in once per device and input type
        static std::mutex mu;
        static bool opted[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lk(mu);
        if (!opted[dev]) {
            e = cudaFuncSetAttribute(bias_bwd_rows<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(2 * (2 * kBiasBwdMaxN - 1) * sizeof(float)));
            if (e != cudaSuccess) return e;
            opted[dev] = true;
        }
    }
    cudaError_t e = cudaMemsetAsync(p.G, 0, (size_t)a.H * nb * sizeof(float), s);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((a.n + kWarps - 1) / kWarps), (unsigned)(a.B * a.H));
    bias_bwd_rows<T><<<grid, kThreads, rows_smem, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bias_bwd_keys<T><<<grid, kThreads, keys_smem, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    unsigned pgrid = (unsigned)a.H;
    size_t psmem = 0;
    if (a.kind == kBiasBuckets) {
        psmem = (size_t)a.num_buckets * sizeof(float);
    } else if (a.kind == kBiasTable) {
        pgrid = a.head_stride == 0 ? 1u : (unsigned)a.H;
        const int lo = a.radius - (a.n - 1) > 0 ? a.radius - (a.n - 1) : 0;
        const int hi = a.radius + (a.n - 1) < 2 * a.radius ? a.radius + (a.n - 1) : 2 * a.radius;
        psmem = (size_t)(hi - lo + 1) * sizeof(float);
    }
    bias_bwd_param<T><<<pgrid, kThreads, psmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace bbwd

long long bias_bwd_rec_floats(int B, int H, int n) {
    // per-row records, rounded up to 64 floats so that G starts 256-byte aligned
    return ((3LL * B * H * n) + 63) / 64 * 64;
}

unsigned long long bias_bwd_workspace_bytes(int B, int H, int n) {
    return (unsigned long long)(bias_bwd_rec_floats(B, H, n) + (long long)H * (2LL * n - 1)) *
           sizeof(float);
}

cudaError_t launch_bias_bwd(const BiasBwdArgs &a, const T5Buckets *t5, cudaStream_t s) {
    if (a.n > kBiasBwdMaxN || a.d > 32 * bbwd::kMaxPer) return cudaErrorNotSupported;
    if (a.H <= 0) return cudaSuccess;
    if (a.n <= 0 || a.B <= 0) {  // no pair: the parameter's gradient is zero
        long long cnt = a.kind == kBiasAlibi ? a.H
                        : a.kind == kBiasBuckets ? (long long)a.num_buckets * a.H
                        : (a.head_stride == 0 ? 0 : (long long)(a.H - 1) * a.head_stride) + 2LL * a.radius + 1;
        return cudaMemsetAsync(a.dbias, 0, (size_t)cnt * sizeof(float), s);
    }
    return a.bf16 ? bbwd::launch_t<__nv_bfloat16>(a, t5, s) : bbwd::launch_t<float>(a, t5, s);
}

}  // namespace relattn
