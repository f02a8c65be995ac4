// Gradients of the Shaw relation-aware attention forward: dq, dk, dv, dw^K, dw^V (and of the
// labelled-edge forward, where a label matrix picks the table row r of each pair in place of
// clip(j - i, k) + k: "Relation-Aware Self-Attention: The Core Modification").
//
// The pages give only the forward pass ("Self-Attention with Relative Position
// Representations" page, section 3.4: eq. 3, eq. 4 and the softmax). The gradients are the
// chain rule through it:
//   dp_ij = dz_i . (v_j + w^V_r),  de_ij = p_ij (dp_ij - D_i),  D_i = sum_j p_ij dp_ij,
//   dq_i = scale sum_j de_ij (k_j + w^K_r),  dk_j = scale sum_i de_ij q_i,
//   dv_j = sum_i p_ij dz_i,  dw^K_r = scale sum_{r_ij = r} de_ij q_i,
//   dw^V_r = sum_{r_ij = r} p_ij dz_i,   r = r_ij = clip(j - i, k) + k.
// As in the forward, the table terms go through per-row quantities of size 2k+1 (never
// n x n x d): R_ir = scale q_i . w^K_r, Rv_ir = dz_i . w^V_r, and the bins
// gamma_ir = sum_{j: r_ij = r} de_ij, beta_ir = sum_{j: r_ij = r} p_ij.
//
// Three kernels, fp32 arithmetic on the SIMT units (inputs bf16 or fp32):
//   rows  one warp per query row: R, Rv, then one pass over the keys for the softmax
//         statistics m, l and D (online, D as a rescaled running sum), then a second pass
//         for dq and the bins; per-row values go to the workspace.
//   keys  one warp per key: dk and dv over the rows that see it, from the per-row values.
//   tabs  one CTA per (head, table row): dw^K and dw^V from the bins (atomic adds when heads
//         share a table).
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "relattn_internal.h"

namespace relattn {
namespace bwd {

constexpr int kWarps = 8;          // rows or keys per CTA
constexpr int kMaxW = 257;         // table rows 2k+1 held per warp in shared memory
constexpr int kMaxPer = 4;         // d <= 128: elements per lane

__device__ __forceinline__ float ld(const float *p, long long i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, long long i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// per-row workspace record: m, l, D, then R[W], Rv[W], gamma[W], beta[W]
__host__ __device__ inline long long rec_floats(int W) { return 3 + 4LL * W; }

template <typename T>
struct Params {
    const T *q, *k, *v, *aK, *aV, *dz;
    long long ths;
    int clip_k, causal;
    int W;                   // table rows: 2k+1, or the number of labels
    const uint8_t *labels;   // labelled edges: row of (i, j) = labels[b * lbs + i * n + j]
    long long lbs;
    int *err;                // device status word (a label without a table row)
    float scale;
    const int *kv_len;
    int B, H, n, d;
    float *dq, *dk, *dv, *daK, *daV;
    float *ws;
};

__device__ __forceinline__ int keys_of(const int *kv_len, int b, int n) {
    return kv_len ? max(0, min(kv_len[b], n)) : n;
}

// table row of pair (i, j): clip(j - i, k) + k, or the pair's label (a label without a
// table row is read as the last row and reported through the status word, as the forward
// does); lab = the row i of the sequence's label matrix
template <typename T>
__device__ __forceinline__ int row_of(const Params<T> &p, const uint8_t *lab, int i, int j) {
    if (!p.labels) return min(p.clip_k, max(-p.clip_k, j - i)) + p.clip_k;
    const int r = lab[j];
    if (r >= p.W) {
        atomicCAS(p.err, 0, kLabelOutOfRange);
        return p.W - 1;
    }
    return r;
}

// ---------------------------------------------------------------------------------- rows
template <typename T>
__global__ void __launch_bounds__(32 * kWarps) bwd_rows(const Params<T> p) {
    __shared__ float sR[kWarps][kMaxW], sRv[kWarps][kMaxW], sG[kWarps][kMaxW], sBe[kWarps][kMaxW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + warp;  // (b*H + h)*n + i
    const long long rows = (long long)p.B * p.H * p.n;
    if (row >= rows) return;
    const int d = p.d, n = p.n, W = p.W;
    const long long bh = row / n;
    const int i = (int)(row - bh * n), b = (int)(bh / p.H), h = (int)(bh % p.H);
    const int nk = keys_of(p.kv_len, b, n);
    const int jend = p.causal ? min(nk, i + 1) : nk;  // keys 0 .. jend-1 are allowed
    const uint8_t *lab = p.labels ? p.labels + (long long)b * p.lbs + (long long)i * n : nullptr;
    float *R = sR[warp], *Rv = sRv[warp], *gam = sG[warp], *bet = sBe[warp];
    float qv[kMaxPer], gv[kMaxPer], acc[kMaxPer];
#pragma unroll
    for (int t = 0; t < kMaxPer; ++t) {
        const int c = lane + 32 * t;
        qv[t] = c < d ? ld(p.q, row * d + c) : 0.f;
        gv[t] = c < d ? ld(p.dz, row * d + c) : 0.f;
        acc[t] = 0.f;
    }
    const long long tab = (long long)h * p.ths;
    for (int r = 0; r < W; ++r) {
        float a = 0.f, bb = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxPer; ++t) {
            const int c = lane + 32 * t;
            if (c < d) {
                if (p.aK) a = fmaf(qv[t], ld(p.aK, tab + (long long)r * d + c), a);
                if (p.aV) bb = fmaf(gv[t], ld(p.aV, tab + (long long)r * d + c), bb);
            }
        }
        a = warp_sum(a);
        bb = warp_sum(bb);
        if (lane == 0) {
            R[r] = p.scale * a;
            Rv[r] = bb;
            gam[r] = 0.f;
            bet[r] = 0.f;
        }
    }
    __syncwarp();
    const long long kv0 = bh * n;  // first key row of this head
    // ---- pass 1: m, l and D = sum p dp (all lanes hold the same values)
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
        const int r = row_of(p, lab, i, j);
        const float e = p.scale * s + R[r];
        const float dp = sv + Rv[r];
        if (e > m) {
            const float a = __expf(m - e);  // 0 when m = -inf
            l *= a;
            S *= a;
            m = e;
        }
        const float pe = __expf(e - m);
        l += pe;
        S = fmaf(pe, dp, S);
    }
    const float D = l > 0.f ? S / l : 0.f;
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    // ---- pass 2: dq and the bins
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
        const int r = row_of(p, lab, i, j);
        const float pr = __expf(p.scale * s + R[r] - m) * inv_l;
        const float de = pr * (sv + Rv[r] - D);
#pragma unroll
        for (int t = 0; t < kMaxPer; ++t) acc[t] = fmaf(p.scale * de, kv[t], acc[t]);
        if (lane == 0) {
            gam[r] += de;
            bet[r] += pr;
        }
    }
    __syncwarp();
    if (p.aK) {  // dq += scale sum_r gamma_r w^K_r
        for (int r = 0; r < W; ++r) {
            const float g = p.scale * gam[r];
#pragma unroll
            for (int t = 0; t < kMaxPer; ++t) {
                const int c = lane + 32 * t;
                if (c < d) acc[t] = fmaf(g, ld(p.aK, tab + (long long)r * d + c), acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kMaxPer; ++t) {
        const int c = lane + 32 * t;
        if (c < d) p.dq[row * d + c] = acc[t];
    }
    float *rec = p.ws + row * rec_floats(W);
    if (lane == 0) {
        rec[0] = m;
        rec[1] = inv_l;
        rec[2] = D;
    }
    for (int r = lane; r < W; r += 32) {
        rec[3 + r] = R[r];
        rec[3 + W + r] = Rv[r];
        rec[3 + 2 * W + r] = gam[r];
        rec[3 + 3 * W + r] = bet[r];
    }
}

// ---------------------------------------------------------------------------------- keys
template <typename T>
__global__ void __launch_bounds__(32 * kWarps) bwd_keys(const Params<T> p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long key = (long long)blockIdx.x * kWarps + warp;  // (b*H + h)*n + j
    const long long rows = (long long)p.B * p.H * p.n;
    if (key >= rows) return;
    const int d = p.d, n = p.n, W = p.W;
    const long long bh = key / n;
    const int j = (int)(key - bh * n), b = (int)(bh / p.H);
    const uint8_t *lab0 = p.labels ? p.labels + (long long)b * p.lbs : nullptr;
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
        const long long q0 = bh * n;
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
            const float *rec = p.ws + (q0 + i) * rec_floats(W);
            // (the row kernel reported an out-of-range label already)
            const int r = p.labels ? min((int)lab0[(long long)i * n + j], W - 1)
                                   : min(p.clip_k, max(-p.clip_k, j - i)) + p.clip_k;
            const float pr = __expf(p.scale * s + rec[3 + r] - rec[0]) * rec[1];
            const float de = pr * (sv + rec[3 + W + r] - rec[2]);
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

// ---------------------------------------------------------------------------------- tables
// block (bh, r): dw^K_r += scale sum_i gamma_ir q_i and dw^V_r += sum_i beta_ir dz_i into the
// head's table (atomic: the batch, and with a shared table all heads, add into one row)
template <typename T>
__global__ void __launch_bounds__(128) bwd_tables(const Params<T> p) {
    const int W = p.W, d = p.d, n = p.n;
    const long long bh = blockIdx.x;
    const int r = blockIdx.y, h = (int)(bh % p.H);
    const long long tab = (long long)h * p.ths + (long long)r * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float ak = 0.f, av = 0.f;
        for (int i = 0; i < n; ++i) {
            const float *rec = p.ws + (bh * n + i) * rec_floats(W);
            if (p.daK) ak = fmaf(rec[3 + 2 * W + r], ld(p.q, (bh * n + i) * d + c), ak);
            if (p.daV) av = fmaf(rec[3 + 3 * W + r], ld(p.dz, (bh * n + i) * d + c), av);
        }
        if (p.daK) atomicAdd(p.daK + tab + c, p.scale * ak);
        if (p.daV) atomicAdd(p.daV + tab + c, av);
    }
}

template <typename T>
cudaError_t launch_t(const BwdArgs &a, cudaStream_t s) {
    Params<T> p;
    p.q = static_cast<const T *>(a.q);
    p.k = static_cast<const T *>(a.k);
    p.v = static_cast<const T *>(a.v);
    p.aK = static_cast<const T *>(a.aK);
    p.aV = static_cast<const T *>(a.aV);
    p.dz = static_cast<const T *>(a.dout);
    p.ths = a.ths;
    p.clip_k = a.clip_k;
    p.causal = a.causal;
    p.W = a.labels ? a.num_labels : 2 * a.clip_k + 1;
    p.labels = a.labels;
    p.lbs = a.lbs;
    p.err = a.err;
    p.scale = a.scale;
    p.kv_len = a.kv_len;
    p.B = a.B;
    p.H = a.H;
    p.n = a.n;
    p.d = a.d;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.daK = a.aK ? a.daK : nullptr;
    p.daV = a.aV ? a.daV : nullptr;
    p.ws = static_cast<float *>(a.workspace);
    const long long rows = (long long)a.B * a.H * a.n;
    const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
    const int W = p.W;
    const int Ht = a.ths == 0 ? 1 : a.H;
    cudaError_t e;
    if (p.daK) {
        e = cudaMemsetAsync(p.daK, 0, (size_t)((Ht - 1) * a.ths + (long long)W * a.d) * sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    if (p.daV) {
        e = cudaMemsetAsync(p.daV, 0, (size_t)((Ht - 1) * a.ths + (long long)W * a.d) * sizeof(float), s);
        if (e != cudaSuccess) return e;
    }
    bwd_rows<T><<<blocks, 32 * kWarps, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_keys<T><<<blocks, 32 * kWarps, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.daK || p.daV) {
        bwd_tables<T><<<dim3((unsigned)(a.B * a.H), (unsigned)W), 128, 0, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace bwd

unsigned long long bwd_simt_workspace_bytes(int B, int H, int n, int W) {
    return (unsigned long long)B * H * n * bwd::rec_floats(W) * sizeof(float);
}

unsigned long long bwd_workspace_bytes(int B, int H, int n, int clip_k) {
    const unsigned long long simt = bwd_simt_workspace_bytes(B, H, n, 2 * clip_k + 1);
    const unsigned long long tc = bwd_tc_workspace_bytes(B, H, n, clip_k);
    return simt > tc ? simt : tc;
}

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t s) {
    const int W = a.labels ? a.num_labels : 2 * a.clip_k + 1;
    if (W > bwd::kMaxW || a.d > 32 * bwd::kMaxPer) return cudaErrorNotSupported;
    if (a.labels && !a.err) return cudaErrorInvalidValue;
    return a.bf16 ? bwd::launch_t<__nv_bfloat16>(a, s) : bwd::launch_t<float>(a, s);
}

}  // namespace relattn
