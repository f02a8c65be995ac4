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
// Without a workspace: one CTA per (sequence, head), 256 threads. The cache is read in chunks
// of kChunk keys:
// each thread computes the logits of its keys (one row of K per thread, 16-byte loads),
// the block takes the chunk's maximum, then the warps accumulate P V with 16-byte loads
// that each cover whole rows of V (d/8 lanes per row, 4 or 2 rows per warp load), with an
// online rescale between chunks. HBM-bound: K and V of the cache are read once.
//
// With a workspace the step runs as a split over all caches at once ("stream-K"): the keys
// of every (sequence, head), laid end to end in (sequence, head, key) order, are cut into one
// equal range per CTA of a grid that fills the GPU once, so every CTA reads the same number of
// cached rows whatever the mix of cache lengths. A CTA walks its range in segments (the part
// of one cache that falls in it); each warp streams groups of keys with the K and V loads of
// a group issued together (and the next group's rows prefetched into L2) and keeps its own
// running maximum, row sum and P V; the warps are merged at the end of a segment, and the
// segment's maximum, row sum and unnormalised P V go to the workspace. A second kernel
// merges the segments of each cache (rescaled to the common maximum) and adds the value bins,
// whose k single-key logits it recomputes from q and the cached keys.
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "relattn_internal.h"

namespace relattn {
namespace decode {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;     // keys whose logits are held in shared memory at a time
constexpr int kMaxBins = 257;    // table rows 0 .. clip_k (clip_k <= 256)
constexpr int kMaxB = 1024;      // sequences of the split (their length prefix sits in shared memory)
constexpr int kMaxGrid = 1024;   // CTAs of the split at most (bounds the workspace)
constexpr bool kPrefetchNext = true;  // split: L2 prefetch of each warp's next group of rows
constexpr long long kMaxKeys = 1LL << 50;  // B * H * T of the split: (key index + 1) * grid stays < 2^63
constexpr unsigned long long kPrefixBytes = ((kMaxB + 1) * 8 + 255) / 256 * 256;
constexpr size_t kMergeStageBytes = 32 * 1024;  // value-table rows the merge stages in shared memory
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    const __nv_bfloat16 *q, *k, *v, *aK, *aV;
    long long ths;        // elements between heads' tables (0: shared)
    int clip_k;
    float scale_log2;     // scale * log2(e)
    const int *cache_len;
    int B, H, T;
    __nv_bfloat16 *out;
    // split: G CTAs; pre[b] = sum of the cache lengths of sequences before b (b = 0 .. B),
    // written by CTA 0 for the merge; part[(c + bh) * (D + 2)] = {max, row sum, P V[D]} of
    // CTA c's segment of cache bh (c + bh is one slot per segment: a CTA's segments are of
    // increasing bh, a cache's of increasing c)
    int G;
    long long *pre;
    float *part;
    int av_staged;  // the merge holds value-table rows 0 .. k in shared memory
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

template <int D, bool AK, bool AV>
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
    const int j_lo = 0, j_hi = t + 1;
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
            if (j >= band0) band[j - band0] = e;  // bin of key j (band0 may be < 0)
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

// ---------------------------------------------------------------------------- split
// Keys of the split are numbered x = H * pre[b] + h * len_b + j (sequence b, head h, key j);
// CTA c of G takes x in [c * total / G, (c + 1) * total / G).
__device__ __forceinline__ long long range_start(long long c, long long total, int G) {
    return c * total / G;
}

// an L2 prefetch of the line holding p
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// q . row over d columns, both bf16 in global memory (16-byte loads, all issued at once)
template <int D>
__device__ __forceinline__ float dot_rows(const __nv_bfloat16 *row, const __nv_bfloat16 *q) {
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row), *q4 = reinterpret_cast<const uint4 *>(q);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 w = __ldg(r4 + c), x = __ldg(q4 + c);
        acc0 = fmaf(bf_lo(w.x), bf_lo(x.x), acc0);
        acc1 = fmaf(bf_hi(w.x), bf_hi(x.x), acc1);
        acc0 = fmaf(bf_lo(w.y), bf_lo(x.y), acc0);
        acc1 = fmaf(bf_hi(w.y), bf_hi(x.y), acc1);
        acc0 = fmaf(bf_lo(w.z), bf_lo(x.z), acc0);
        acc1 = fmaf(bf_hi(w.z), bf_hi(x.z), acc1);
        acc0 = fmaf(bf_lo(w.w), bf_lo(x.w), acc0);
        acc1 = fmaf(bf_hi(w.w), bf_hi(x.w), acc1);
    }
    return acc0 + acc1;
}

template <int D, bool AK>
__global__ void __launch_bounds__(kThreads, 2) relattn_decode_split_kernel(const Params p) {
    // a warp group of keys: 8 loads per lane, each covering KPW whole rows (LPR lanes x 16 B)
    constexpr int LPR = D / 8, KPW = 32 / LPR, NK = 8 * KPW;
    constexpr int PER = kMaxB / kThreads;  // lengths per thread in the prefix scan
    __shared__ long long pre[kMaxB + 1];
    __shared__ long long wsum[kWarps];
    __shared__ float rel[kMaxBins];        // R_r * scale * log2(e) of the current segment
    __shared__ float wm[kWarps], wl[kWarps];
    __shared__ float wacc[kWarps][D];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B, H = p.H;
    // the merge may be scheduled as soon as every CTA of this grid runs (its CTAs fit only
    // where CTAs of this grid have exited; it waits for this grid's results before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- prefix sums of the cache lengths (every CTA; CTA 0 also leaves them for the merge)
    {
        long long v[PER], sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int b = tid * PER + i;
            v[i] = b < B ? min(max(p.cache_len[b], 0), p.T) : 0;
            sum += v[i];
        }
        long long inc = sum;  // inclusive scan over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        long long run = inc - sum;
        for (int w = 0; w < warp; ++w) run += wsum[w];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            pre[tid * PER + i] = run;
            run += v[i];
        }
        if (tid == kThreads - 1) pre[kMaxB] = run;  // entries past B are 0: pre[B..] = total
        __syncthreads();
    }
    if (blockIdx.x == 0)
        for (int b = tid; b <= B; b += kThreads) p.pre[b] = pre[b];
    const long long total = (long long)H * pre[B];
    const long long x1 = range_start(blockIdx.x + 1, total, p.G);
    long long x = range_start(blockIdx.x, total, p.G);
    const int ks = lane / LPR, cg = lane % LPR;  // key of a warp load, 8-column group

    while (x < x1) {
        // ---- the segment: sequence b with H * pre[b] <= x < H * pre[b + 1] (never empty)
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long long)H * pre[mid] <= x) lo = mid;
            else hi = mid;
        }
        const int b = lo;
        const int len = (int)(pre[b + 1] - pre[b]);
        const long long r0 = x - (long long)H * pre[b];
        const int h = (int)(r0 / len);
        const int j0 = (int)(r0 - (long long)h * len);
        const int j1 = (int)min((long long)len, (long long)j0 + (x1 - x));
        const int bh = b * H + h, seg = j1 - j0;
        const int band0 = len - 1 - p.clip_k;  // keys j <= band0 take table row 0
        x += seg;

        const __nv_bfloat16 *qrow = p.q + (long long)bh * D;
        if (AK) {  // the table rows this segment reads: 0 .. max(0, j1 - 1 - band0)
            const __nv_bfloat16 *tab = p.aK + (long long)h * p.ths;
            const int rmax = max(0, j1 - 1 - band0);
            for (int r = tid; r <= rmax; r += kThreads)
                rel[r] = dot_rows<D>(tab + (long long)r * D, qrow) * p.scale_log2;
        }
        float qr[8];  // this lane's 8 columns of q * scale * log2(e)
        {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(qrow) + cg);
            qr[0] = bf_lo(w.x) * p.scale_log2;
            qr[1] = bf_hi(w.x) * p.scale_log2;
            qr[2] = bf_lo(w.y) * p.scale_log2;
            qr[3] = bf_hi(w.y) * p.scale_log2;
            qr[4] = bf_lo(w.z) * p.scale_log2;
            qr[5] = bf_hi(w.z) * p.scale_log2;
            qr[6] = bf_lo(w.w) * p.scale_log2;
            qr[7] = bf_hi(w.w) * p.scale_log2;
        }
        if (AK) __syncthreads();
        const long long row0 = (long long)bh * p.T + j0;  // first cached row of the segment
        const uint4 *kb = reinterpret_cast<const uint4 *>(p.k + row0 * D) + cg;
        const uint4 *vb = reinterpret_cast<const uint4 *>(p.v + row0 * D) + cg;
        float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = 0.f;
        // ---- warp groups of NK keys: K and V loads of the group first (and an L2 prefetch of
        // the warp's next group), then the logits, the group maximum, the rescale and P V
        // (keys past the segment load its last row and get probability 0)
        for (int g0 = warp * NK; g0 < seg; g0 += kWarps * NK) {
            uint4 kw[8], vw[8];
            int u_of[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                u_of[u] = g0 + u * KPW + ks;
                kw[u] = __ldg(kb + (long long)min(u_of[u], seg - 1) * LPR);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) vw[u] = __ldg(vb + (long long)min(u_of[u], seg - 1) * LPR);
            if (kPrefetchNext && g0 + kWarps * NK < seg && lane < NK) {  // the next group: a row per lane
                const int nxt = min(g0 + kWarps * NK + lane, seg - 1);
#pragma unroll
                for (int hl = 0; hl < D / 64; ++hl) {  // the 128-byte lines of the row
                    prefetch_l2(kb - cg + (long long)nxt * LPR + 8 * hl);
                    prefetch_l2(vb - cg + (long long)nxt * LPR + 8 * hl);
                }
            }
            float e[8], gmax = -INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint4 w = kw[u];
                float a0 = bf_lo(w.x) * qr[0], a1 = bf_hi(w.x) * qr[1];
                a0 = fmaf(bf_lo(w.y), qr[2], a0);
                a1 = fmaf(bf_hi(w.y), qr[3], a1);
                a0 = fmaf(bf_lo(w.z), qr[4], a0);
                a1 = fmaf(bf_hi(w.z), qr[5], a1);
                a0 = fmaf(bf_lo(w.w), qr[6], a0);
                a1 = fmaf(bf_hi(w.w), qr[7], a1);
                float sdot = a0 + a1;
#pragma unroll
                for (int o = 1; o < LPR; o <<= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, o);
                if (AK) sdot += rel[max(0, j0 + min(u_of[u], seg - 1) - band0)];
                e[u] = u_of[u] < seg ? sdot : -INFINITY;
                gmax = fmaxf(gmax, e[u]);
            }
#pragma unroll
            for (int o = LPR; o < 32; o <<= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
            if (gmax > m) {  // warp-uniform; the first group always rescales (from nothing)
                const float alpha = exp2f(m - gmax);
                m = gmax;
                l *= alpha;
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c] *= alpha;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float pj = exp2f(e[u] - m);
                const uint4 w = vw[u];
                acc[0] = fmaf(pj, bf_lo(w.x), acc[0]);
                acc[1] = fmaf(pj, bf_hi(w.x), acc[1]);
                acc[2] = fmaf(pj, bf_lo(w.y), acc[2]);
                acc[3] = fmaf(pj, bf_hi(w.y), acc[3]);
                acc[4] = fmaf(pj, bf_lo(w.z), acc[4]);
                acc[5] = fmaf(pj, bf_hi(w.z), acc[5]);
                acc[6] = fmaf(pj, bf_lo(w.w), acc[6]);
                acc[7] = fmaf(pj, bf_hi(w.w), acc[7]);
                if (cg == 0) l += pj;
            }
        }
        // ---- merge: the KPW keys of a warp load (same m), then the warps (rescaled)
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], o);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (ks == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c) wacc[warp][8 * cg + c] = acc[c];
        }
        if (lane == 0) {
            wm[warp] = m;  // -inf for a warp without keys: weight 0 below
            wl[warp] = l;
        }
        __syncthreads();
        float *part = p.part + ((long long)blockIdx.x + bh) * (D + 2);
        if (tid < D) {
            float M = wm[0];  // warp 0 always has keys
#pragma unroll
            for (int w = 1; w < kWarps; ++w) M = fmaxf(M, wm[w]);
            float o = 0.f, L = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float sc = exp2f(wm[w] - M);
                o = fmaf(wacc[w][tid], sc, o);
                L = fmaf(wl[w], sc, L);
            }
            part[2 + tid] = o;
            if (tid == 0) {
                part[0] = M;
                part[1] = L;
            }
        }
        __syncthreads();  // the shared state is rewritten by the next segment
    }
}

// The segments of one cache: their maxima, row sums and P V merged online (each output thread
// walks the same segments in the same order, so all reach the same maximum M and sum L),
// then the value bins (keys t-k+1 .. t one each, bin 0 what the row sum leaves) and the
// normalisation. It is launched as a programmatic dependent of the split kernel: what reads
// only the step's inputs (the bins' logits, the value-table rows) runs before the wait for
// the split kernel's results.
template <int D, bool AK, bool AV>
__global__ void __launch_bounds__(128) relattn_decode_merge(const Params p) {
    extern __shared__ __align__(16) unsigned char av_rows[];  // aV rows 0 .. k (bf16), if staged
    __shared__ float band[kMaxBins];  // logits of bins 1 .. k (log2 domain)
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H, tid = threadIdx.x;
    const int len = min(max(p.cache_len[b], 0), p.T);
    __nv_bfloat16 *orow = p.out + (long long)bh * D;
    if (len == 0) {
        for (int c = tid; c < D; c += 128) orow[c] = __float2bfloat16(0.f);
        return;
    }
    const int t = len - 1, k = p.clip_k, band0 = t - k;
    const int r_lo = max(1, -band0);  // bins 1 .. k whose key j = band0 + r exists
    const long long tab = (long long)h * p.ths;
    const __nv_bfloat16 *wv = AV ? p.aV + tab : nullptr;
    if (AV) {
        const __nv_bfloat16 *qrow = p.q + (long long)bh * D;
        const __nv_bfloat16 *kbase = p.k + (long long)bh * p.T * D;
        for (int r = r_lo + tid; r <= k; r += 128) {
            float e = dot_rows<D>(kbase + (long long)(band0 + r) * D, qrow);
            if (AK) e += dot_rows<D>(p.aK + tab + (long long)r * D, qrow);
            band[r] = e * p.scale_log2;
        }
        if (p.av_staged) {
            const int n16 = (k + 1) * (D / 8);
            for (int i = tid; i < n16; i += 128)
                reinterpret_cast<uint4 *>(av_rows)[i] = __ldg(reinterpret_cast<const uint4 *>(wv) + i);
            wv = reinterpret_cast<const __nv_bfloat16 *>(av_rows);
        }
    }
    // the split kernel's prefix and segment records from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // CTA of key x: the largest c with c * total / G <= x, i.e. ((x + 1) G - 1) / total
    const long long total = (long long)p.H * p.pre[p.B];
    const long long xf = (long long)p.H * p.pre[b] + (long long)h * len;
    const int c0 = (int)(((xf + 1) * p.G - 1) / total);
    const int c1 = (int)(((xf + len) * p.G - 1) / total);
    // CTAs c0 .. c1, slots c0 + bh .. c1 + bh; with fewer keys than CTAs some CTAs in between
    // own no key and wrote nothing: their slots are skipped
    const int np = c1 - c0 + 1;
    const float *part = p.part + ((long long)c0 + bh) * (D + 2);
    __syncthreads();  // band[] and the staged rows
    for (int c = tid; c < D; c += 128) {
        float M = -INFINITY, L = 0.f, o = 0.f;
#pragma unroll 2
        for (int i = 0; i < np; ++i) {
            const float *rec = part + (long long)i * (D + 2);
            const float mi = rec[0], li = rec[1], oi = rec[2 + c];
            if (range_start(c0 + i, total, p.G) == range_start(c0 + i + 1, total, p.G)) continue;
            if (mi > M) {  // rescale what was merged so far (nothing on the first segment)
                const float a = exp2f(M - mi);
                L *= a;
                o *= a;
                M = mi;
            }
            const float w = exp2f(mi - M);
            L = fmaf(li, w, L);
            o = fmaf(oi, w, o);
        }
        if (AV) {
            float s_band = 0.f, ov = 0.f;
#pragma unroll 4
            for (int r = r_lo; r <= k; ++r) {
                const float pr = exp2f(band[r] - M);
                s_band += pr;
                ov = fmaf(pr, __bfloat162float(wv[(long long)r * D + c]), ov);
            }
            o += fmaf(fmaxf(0.f, L - s_band), __bfloat162float(wv[c]), ov);
        }
        orow[c] = __float2bfloat16(o / L);
    }
}

// CTAs of the split: every SM filled once (the kernel's resident CTAs per SM), at most kMaxGrid
template <int D, bool AK>
int split_grid() {
    static int cache[64][2] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    int &g = cache[dev][AK ? 1 : 0];
    if (g == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, relattn_decode_split_kernel<D, AK>,
                                                          kThreads, 0) != cudaSuccess)
            return 0;
        g = min(kMaxGrid, max(1, sms * per_sm));
    }
    return g;
}

template <int D, bool AK, bool AV>
cudaError_t launch_variant(Params p, bool split, cudaStream_t s) {
    if (!split) {
        relattn_decode_kernel<D, AK, AV><<<dim3((unsigned)(p.B * p.H)), kThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    p.G = split_grid<D, AK>();
    if (p.G <= 0) return cudaErrorUnknown;
    relattn_decode_split_kernel<D, AK><<<dim3((unsigned)p.G), kThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the merge as a programmatic dependent launch on the same stream
    const size_t av_bytes = (size_t)(p.clip_k + 1) * D * sizeof(__nv_bfloat16);
    p.av_staged = AV && av_bytes <= kMergeStageBytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.H));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = p.av_staged ? av_bytes : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, relattn_decode_merge<D, AK, AV>, p);
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
    const unsigned long long need = decode_workspace_bytes(a.B, a.H, a.T, a.d);
    const bool split = need > 0 && a.workspace && a.workspace_bytes >= need;
    p.G = 0;
    p.av_staged = 0;
    p.pre = split ? static_cast<long long *>(a.workspace) : nullptr;
    p.part = split ? reinterpret_cast<float *>(static_cast<char *>(a.workspace) + kPrefixBytes) : nullptr;
    if (a.aK && a.aV) return launch_variant<D, true, true>(p, split, s);
    if (a.aK) return launch_variant<D, true, false>(p, split, s);
    if (a.aV) return launch_variant<D, false, true>(p, split, s);
    return launch_variant<D, false, false>(p, split, s);
}

}  // namespace decode

unsigned long long decode_workspace_bytes(int B, int H, int T, int d) {
    // the split needs the sequences' length prefix in shared memory and key indices whose
    // product with the grid fits 63 bits; past that the single-pass kernel runs
    if (B > decode::kMaxB || (long long)B * H * T > decode::kMaxKeys) return 0;
    return decode::kPrefixBytes +
           (unsigned long long)(decode::kMaxGrid + (long long)B * H) * (d + 2) * sizeof(float);
}

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
    if (a.clip_k + 1 > decode::kMaxBins) return cudaErrorNotSupported;
    return a.d == 64 ? decode::launch_d<64>(a, s) : decode::launch_d<128>(a, s);
}

}  // namespace relattn
