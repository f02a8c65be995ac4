// One incremental decoding step of a causal decoder with Shaw relative terms: the new
// token's query against its sequence's key/value cache.
//
// Paper summary page, section 3.4 (eq. 3 and eq. 4, clip(j - i, k)): for the token at
// position t = cache_len - 1, e_j = scale * q . (k_j + w^K_{clip(j - t, k)}) over j = 0 .. t,
// and z = sum_j softmax(e)_j (v_j + w^V_{clip(j - t, k)}). Only table rows 0 .. k (offsets
// -k .. 0) are ever used. As in the forward kernels the key term goes through R_r = q . w^K_r
// (one dot product per table row) and the value term through bins beta_r (keys at offset
// <= -k share bin 0; each of the last k keys has its own bin), so the sum over the cache
// reads each cached row once and nothing of size cache x d is built.
//
// One CTA per (sequence, head), 256 threads. The cache is read in chunks of kChunk keys:
// each thread computes the logits of its keys (one row of K per thread, 16-byte loads),
// the block takes the chunk's maximum, then the warps accumulate P V with 16-byte loads
// that each cover whole rows of V (d/8 lanes per row, 4 or 2 rows per warp load), with an
// online rescale between chunks. HBM-bound: K and V of the cache are read once.
//
// With few heads (at most kSplitMaxHeads) and a workspace the cache of a head is split into
// pieces of kSplit keys, one CTA each (grid x = heads, y = pieces), so that a small batch
// still fills the GPU; each piece writes its maximum, row sum and unnormalised P V into the
// workspace, and
// a second kernel combines the pieces of a head (rescaled to the common maximum) and adds
// the value bins, whose k single-key logits it recomputes from q and the cached keys.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "relattn_internal.h"

namespace relattn {
namespace decode {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;     // keys whose logits are held in shared memory at a time
constexpr int kMaxBins = 257;    // table rows 0 .. clip_k (clip_k <= 256)
constexpr int kSplit = 512;      // keys per CTA with a workspace
constexpr int kSplitMaxHeads = 256;  // more heads than this fill the GPU without a split
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    const __nv_bfloat16 *q, *k, *v, *aK, *aV;
    long long ths;        // elements between heads' tables (0: shared)
    int clip_k;
    float scale_log2;     // scale * log2(e)
    const int *cache_len;
    int B, H, T;
    __nv_bfloat16 *out;
    float *ws;   // workspace: per (head, piece) {max, row sum, P V[D]}, or null
    int npiece;  // pieces per head with a workspace
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D>
__device__ __forceinline__ float dot_row(const __nv_bfloat16 *row, const float *qs) {
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 w = __ldg(r4 + c);
        acc0 = fmaf(bf_lo(w.x), qs[8 * c + 0], acc0);
        acc1 = fmaf(bf_hi(w.x), qs[8 * c + 1], acc1);
        acc0 = fmaf(bf_lo(w.y), qs[8 * c + 2], acc0);
        acc1 = fmaf(bf_hi(w.y), qs[8 * c + 3], acc1);
        acc0 = fmaf(bf_lo(w.z), qs[8 * c + 4], acc0);
        acc1 = fmaf(bf_hi(w.z), qs[8 * c + 5], acc1);
        acc0 = fmaf(bf_lo(w.w), qs[8 * c + 6], acc0);
        acc1 = fmaf(bf_hi(w.w), qs[8 * c + 7], acc1);
    }
    return acc0 + acc1;
}

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

template <int D, bool AK, bool AV, bool SPLIT>
__global__ void __launch_bounds__(kThreads) relattn_decode_kernel(const Params p) {
    // P V: a row of V is LPR lanes x 16 bytes; a warp load covers KPW keys
    constexpr int LPR = D / 8, KPW = 32 / LPR;
    __shared__ float qs[D];                 // q * scale * log2(e)
    __shared__ float rel[kMaxBins];         // R_r * scale * log2(e), r = 0 .. k
    __shared__ float e_s[kChunk];           // logits of the chunk (log2 domain)
    __shared__ float band[kMaxBins];        // logits of the last k + 1 keys (bins 0 .. k)
    __shared__ float red[kWarps];
    __shared__ float acc_s[kWarps][D];
    __shared__ float lw_s[kWarps];

    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int len = min(max(p.cache_len[b], 0), p.T);
    __nv_bfloat16 *orow = p.out + (long long)bh * D;
    if (len == 0) {  // no key: zeros
        for (int c = tid; c < D; c += kThreads) orow[c] = __float2bfloat16(0.f);
        return;
    }
    const int t = len - 1, k = p.clip_k;
    const int band0 = t - k;  // keys j >= band0 + 1 have their own bin, j <= band0 share bin 0
    // keys of this CTA: the whole cache, or piece blockIdx.y of kSplit keys
    const int j_lo = SPLIT ? (int)blockIdx.y * kSplit : 0;
    const int j_hi = SPLIT ? min(t + 1, j_lo + kSplit) : t + 1;
    float *part = SPLIT ? p.ws + ((long long)bh * p.npiece + blockIdx.y) * (D + 2) : nullptr;
    if (SPLIT && j_lo >= j_hi) {  // past the end of this cache: an empty piece
        if (tid == 0) {
            part[0] = -INFINITY;
            part[1] = 0.f;
        }
        for (int c = tid; c < D; c += kThreads) part[2 + c] = 0.f;
        return;
    }
    const __nv_bfloat16 *qrow = p.q + (long long)bh * D;
    for (int c = tid; c < D; c += kThreads) qs[c] = __bfloat162float(qrow[c]) * p.scale_log2;
    __syncthreads();
    const long long tab = (long long)h * p.ths;
    if (AK) {
        for (int r = tid; r <= k; r += kThreads) rel[r] = dot_row<D>(p.aK + tab + (long long)r * D, qs);
    }
    __syncthreads();

    const __nv_bfloat16 *kbase = p.k + (long long)bh * p.T * D;
    const __nv_bfloat16 *vbase = p.v + (long long)bh * p.T * D;
    float m = -INFINITY, lw = 0.f;  // running maximum; this lane's share of the row sum
    const int ks = lane / LPR, cg = lane % LPR;  // key of the warp load, 8-column group
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;

    for (int j0 = j_lo; j0 < j_hi; j0 += kChunk) {
        const int cnt = min(kChunk, j_hi - j0);
        // ---- logits of the chunk, one cached key row per thread
        float tmax = -INFINITY;
        for (int u = tid; u < cnt; u += kThreads) {
            const int j = j0 + u;
            float e = dot_row<D>(kbase + (long long)j * D, qs);
            if (AK) e += rel[max(0, j - band0)];
            e_s[u] = e;
            if (!SPLIT && j >= band0) band[j - band0] = e;  // bin of key j (band0 may be < 0)
            tmax = fmaxf(tmax, e);
        }
        const float cmax = block_max(tmax, red);  // also orders the e_s writes before reads
        // ---- online rescale (every warp holds the same m)
        const float m_new = fmaxf(m, cmax);
        const float alpha = exp2f(m - m_new);  // 0 on the first chunk
        m = m_new;
        lw *= alpha;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] *= alpha;
        // ---- P V: warp w takes keys w*KPW + ks, then every kWarps*KPW-th; lane cg owns
        // columns 8cg .. 8cg+7 of its key's row (16-byte loads, KPW whole rows per load)
#pragma unroll 8
        for (int u = warp * KPW + ks; u < cnt; u += kWarps * KPW) {
            const float pj = exp2f(e_s[u] - m);
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(vbase + (long long)(j0 + u) * D) + cg);
            acc[0] = fmaf(pj, bf_lo(w.x), acc[0]);
            acc[1] = fmaf(pj, bf_hi(w.x), acc[1]);
            acc[2] = fmaf(pj, bf_lo(w.y), acc[2]);
            acc[3] = fmaf(pj, bf_hi(w.y), acc[3]);
            acc[4] = fmaf(pj, bf_lo(w.z), acc[4]);
            acc[5] = fmaf(pj, bf_hi(w.z), acc[5]);
            acc[6] = fmaf(pj, bf_lo(w.w), acc[6]);
            acc[7] = fmaf(pj, bf_hi(w.w), acc[7]);
            if (cg == 0) lw += pj;
        }
        __syncthreads();  // e_s is rewritten by the next chunk
    }
    // ---- combine: the KPW key groups of a warp (lanes cg, cg + LPR, ...), then the warps
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], o);
        lw += __shfl_xor_sync(0xffffffffu, lw, o);
    }
    if (ks == 0) {
#pragma unroll
        for (int c = 0; c < 8; ++c) acc_s[warp][8 * cg + c] = acc[c];
    }
    if (lane == 0) lw_s[warp] = lw;
    __syncthreads();
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) l += lw_s[w];
    if (SPLIT) {  // this piece's maximum, row sum and unnormalised P V
        if (tid == 0) {
            part[0] = m;
            part[1] = l;
        }
        for (int c = tid; c < D; c += kThreads) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) o += acc_s[w][c];
            part[2 + c] = o;
        }
        return;
    }
    const float inv = 1.f / l;
    for (int c = tid; c < D; c += kThreads) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) o += acc_s[w][c];
        if (AV) {
            // bins 1 .. k: one key each (offsets -k+1 .. 0); bin 0: the rest of the row sum
            const __nv_bfloat16 *wv = p.aV + tab;
            float s_band = 0.f, ov = 0.f;
            for (int r = 1; r <= k; ++r) {
                const int j = band0 + r;
                if (j < 0) continue;
                const float pr = exp2f(band[r] - m);
                s_band += pr;
                ov = fmaf(pr, __bfloat162float(wv[(long long)r * D + c]), ov);
            }
            const float b0 = fmaxf(0.f, l - s_band);
            ov = fmaf(b0, __bfloat162float(wv[c]), ov);
            o += ov;
        }
        orow[c] = __float2bfloat16(o * inv);
    }
}

// The pieces of one head: common maximum M, row sum and P V rescaled to it, then the value
// bins (keys t-k+1 .. t one each, bin 0 what the row sum leaves) and the normalisation.
template <int D, bool AK, bool AV>
__global__ void __launch_bounds__(128) relattn_decode_combine(const Params p) {
    __shared__ float qs[D];
    __shared__ float band[kMaxBins];
    __shared__ float scl[64];
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H, tid = threadIdx.x;
    const int len = min(max(p.cache_len[b], 0), p.T);
    __nv_bfloat16 *orow = p.out + (long long)bh * D;
    if (len == 0) {
        for (int c = tid; c < D; c += 128) orow[c] = __float2bfloat16(0.f);
        return;
    }
    const int t = len - 1, k = p.clip_k, band0 = t - k;
    const int np = min(p.npiece, (t + kSplit) / kSplit);  // pieces holding keys
    const float *part = p.ws + (long long)bh * p.npiece * (D + 2);
    float M = -INFINITY;
    for (int i = 0; i < np; ++i) M = fmaxf(M, part[(long long)i * (D + 2)]);
    if (tid < np && tid < 64) scl[tid] = exp2f(part[(long long)tid * (D + 2)] - M);
    const __nv_bfloat16 *qrow = p.q + (long long)bh * D;
    for (int c = tid; c < D; c += 128) qs[c] = __bfloat162float(qrow[c]) * p.scale_log2;
    __syncthreads();
    float L = 0.f;
    for (int i = 0; i < np; ++i)
        L = fmaf(part[(long long)i * (D + 2) + 1], i < 64 ? scl[i] : exp2f(part[(long long)i * (D + 2)] - M), L);
    const long long tab = (long long)h * p.ths;
    if (AV) {  // logits of the single-key bins 1 .. k (keys band0 + 1 .. t)
        const __nv_bfloat16 *kbase = p.k + (long long)bh * p.T * D;
        for (int r = 1 + tid; r <= k; r += 128) {
            const int j = band0 + r;
            if (j < 0) continue;
            float e = dot_row<D>(kbase + (long long)j * D, qs);
            if (AK) e += dot_row<D>(p.aK + tab + (long long)r * D, qs);
            band[r] = e;
        }
    }
    __syncthreads();
    const float inv = 1.f / L;
    for (int c = tid; c < D; c += 128) {
        float o = 0.f;
        for (int i = 0; i < np; ++i)
            o = fmaf(part[(long long)i * (D + 2) + 2 + c], i < 64 ? scl[i] : exp2f(part[(long long)i * (D + 2)] - M), o);
        if (AV) {
            const __nv_bfloat16 *wv = p.aV + tab;
            float s_band = 0.f, ov = 0.f;
            for (int r = 1; r <= k; ++r) {
                if (band0 + r < 0) continue;
                const float pr = exp2f(band[r] - M);
                s_band += pr;
                ov = fmaf(pr, __bfloat162float(wv[(long long)r * D + c]), ov);
            }
            ov = fmaf(fmaxf(0.f, L - s_band), __bfloat162float(wv[c]), ov);
            o += ov;
        }
        orow[c] = __float2bfloat16(o * inv);
    }
}

template <int D, bool AK, bool AV>
cudaError_t launch_variant(const Params &p, bool split, cudaStream_t s) {
    if (!split) {
        relattn_decode_kernel<D, AK, AV, false><<<dim3((unsigned)(p.B * p.H)), kThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    relattn_decode_kernel<D, AK, AV, true>
        <<<dim3((unsigned)(p.B * p.H), (unsigned)p.npiece), kThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    relattn_decode_combine<D, AK, AV><<<dim3((unsigned)(p.B * p.H)), 128, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs &a, cudaStream_t s) {
    Params p;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k = static_cast<const __nv_bfloat16 *>(a.k_cache);
    p.v = static_cast<const __nv_bfloat16 *>(a.v_cache);
    p.aK = static_cast<const __nv_bfloat16 *>(a.aK);
    p.aV = static_cast<const __nv_bfloat16 *>(a.aV);
    p.ths = a.ths;
    p.clip_k = a.clip_k;
    p.scale_log2 = a.scale * kLog2e;
    p.cache_len = a.cache_len;
    p.B = a.B;
    p.H = a.H;
    p.T = a.T;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.npiece = (a.T + kSplit - 1) / kSplit;
    const unsigned long long need = decode_workspace_bytes(a.B, a.H, a.T, a.d);
    const bool split = need > 0 && a.workspace && a.workspace_bytes >= need;
    p.ws = split ? static_cast<float *>(a.workspace) : nullptr;
    if (a.aK && a.aV) return launch_variant<D, true, true>(p, split, s);
    if (a.aK) return launch_variant<D, true, false>(p, split, s);
    if (a.aV) return launch_variant<D, false, true>(p, split, s);
    return launch_variant<D, false, false>(p, split, s);
}

}  // namespace decode

unsigned long long decode_workspace_bytes(int B, int H, int T, int d) {
    const long long pieces = (T + decode::kSplit - 1) / decode::kSplit;
    // one piece, or enough heads to fill the GPU: the single-pass kernel needs nothing (with
    // 512 heads of 1K-2K keys it measured faster than the split)
    if (pieces <= 1 || (long long)B * H > decode::kSplitMaxHeads) return 0;
    return (unsigned long long)B * H * pieces * (d + 2) * sizeof(float);
}

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
    if (a.clip_k + 1 > decode::kMaxBins) return cudaErrorNotSupported;
    return a.d == 64 ? decode::launch_d<64>(a, s) : decode::launch_d<128>(a, s);
}

}  // namespace relattn
