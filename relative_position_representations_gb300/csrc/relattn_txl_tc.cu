// Transformer-XL relative attention on the tensor cores (bf16 in, fp32 accumulate, head
// dimension 64 or 128). Method: "Relative Position Encoding in Transformer-XL" page (the
// four-term score and the roles of the global biases u and v) and "Relative position
// embeddings" page, section "Transformer-XL":
//   A_ij = q_i.k_j + q_i.r_ij + u.k_j + v.r_ij,    r_ij = rel[h][(j - i) + n - 1]
//   z_i  = sum_j softmax_j(scale * A)_ij v_j
//
// One CTA per (head, 128-row query tile), longest causal rows first. Per key tile of 128 keys:
//   S = Q K^T                     (tcgen05, M = 128, N = 128)   terms (a)
//   T = Q R_win^T                 (tcgen05, M = 128, N = 256)   term (b) for every offset the
//                                 tile pair spans: R_win is rel rows (j0 - i0 - 127) + n - 1
//                                 onward, 256 of them (a TMA box that may start before row 0
//                                 or run past the end; those rows read as zero)
//   u.k_j and v.r_o               per-key and per-offset scalars, terms (c) and (d), fp32 dot
//                                 products by the row threads from the staged K and R_win rows
//   O += P V                      (tcgen05, P bf16 over the S columns)
// Element (i, j) of T sits in column (j - i) + 127 of row i: a diagonal. The row thread loads
// the 64 columns its warp's rows need for a chunk of 32 keys into registers, adds v.r, and
// stores them to its own row of a shared-memory scratch (64 floats + 4 of padding, so that
// the 32 lanes' stores and their skewed reads each hit distinct banks); it then reads column
// (t - lane + 31) for key t of the chunk, the diagonal, from its own row.
// Softmax in the exp2 domain with a lazy rescale of O (only when the row maximum grows by
// more than 2^8), one thread per query row (TMEM lane = row).
// Roles (192 threads): warp 0 TMA loads (Q, then K, V, R_win per key tile into a ring),
// warp 1 MMA issue (one elected lane), warps 2-5 the query rows.
// Every wait is bounded; a wait that runs out sets the device status word and the CTA drains
// and exits.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "relattn_internal.h"
#include "relattn_tc_launch.cuh"

namespace relattn {
namespace txltc {

using tc::BM;
using tc::BN;
using tc::kLog2e;
using tc::Shared;

constexpr int kRowWarp0 = 2;
// row groups: d = 64 runs two threads per row (each half of a tile's keys), d = 128 one (the
// per-thread diagonal scratch of two groups would not fit beside its tiles)
template <int D> struct Groups {
    static constexpr int NG = D == 64 ? 2 : 1;
    static constexpr int kRowThreads = 128 * NG;
    static constexpr int kThreads = 64 + kRowThreads;  // warp 0 TMA, warp 1 MMA issue, row warps
    static constexpr int CPT = 4 / NG;                  // 32-key chunks per thread and tile
};
constexpr int kWin = 256;       // R_win rows per key tile (the 255 offsets of a tile pair, + 1)
constexpr int kSkew = 68;       // floats per row of the diagonal scratch
constexpr int kMaxStages = 2;
constexpr float kRescaleLog2 = 8.0f;

struct Params {
    int BH, H, n, n_tiles, causal, shared;
    float c;                          // scale * log2(e)
    const int *kv_len;
    int *err;
    const __nv_bfloat16 *u, *vb;      // [H|1, d]
    __nv_bfloat16 *out;               // [B, H, n, d]
    uint32_t off_q, off_k, off_v, off_r, off_skew, off_uk, off_vr, off_uv, off_x, off_bar;
    uint32_t stage_kv, stage_r;       // bytes per stage: one K (or V) tile, one R_win tile
    int stages;
    long long wait_limit;
};

enum : int {
    X_Q = 0, X_S_FULL, X_S_EMPTY, X_P_FULL, X_PV_DONE, X_DRAIN,
    X_KV_FULL = 6, X_KV_EMPTY = X_KV_FULL + kMaxStages, kBars = X_KV_EMPTY + kMaxStages
};

__device__ __forceinline__ uint64_t kstep(int kk, int rows) {
    return (uint64_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t mnstep(int kk) { return (uint64_t)(kk * 16 * 128 >> 4); }

// dot product of a bf16 row of a 128-byte-swizzled tile (row `row`, 64-column blocks
// `block_bytes` apart) with an fp32 vector in shared memory
template <int D>
__device__ __forceinline__ float swz_dot(const uint8_t *tile, uint32_t block_bytes, int row, const float *w) {
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
        const uint8_t *r = tile + h * block_bytes + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 x = *reinterpret_cast<const uint4 *>(r + (((uint32_t)c ^ ((uint32_t)row & 7u)) << 4));
            const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
            const float *ww = w + 64 * h + 8 * c;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(ptx::bf16lo_to_f32(wv[e]), ww[2 * e], acc);
                acc = fmaf(ptx::bf16hi_to_f32(wv[e]), ww[2 * e + 1], acc);
            }
        }
    }
    return acc;
}

template <int D>
__global__ void __launch_bounds__(Groups<D>::kThreads, 1)
    txl_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
                  const __grid_constant__ Params p) {
    // d = 64: P has its own TMEM columns, so the next tile's S and T run during this tile's
    // softmax; d = 128: P over S (TMEM is full), the next S waits for this P V
    constexpr bool P_OWN = D == 64;
    constexpr int NG = Groups<D>::NG, CPT = Groups<D>::CPT, kRowThreads = Groups<D>::kRowThreads;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    Shared sh;
    sh.base = (raw + 1023u) & ~1023u;
    sh.ptr = smem_raw + (sh.base - raw);
    sh.abort_flag = reinterpret_cast<volatile int *>(sh.ptr + p.off_bar + 8 * 32 + 4);
    sh.limit = p.wait_limit;
    const uint32_t bar0 = sh.base + p.off_bar;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = p.n_tiles - 1 - (int)blockIdx.x / p.BH, bh = (int)blockIdx.x % p.BH;
    const int i0 = qt * BM;
    const int nk = p.kv_len ? max(0, min(p.kv_len[bh / p.H], p.n)) : p.n;
    const int nkc = p.causal ? min(nk, i0 + BM) : nk;
    const int J = (nkc + BN - 1) / BN;
    const int th = p.shared ? 0 : bh % p.H;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kBars; ++i)
            ptx::mbar_init(bar(i), (i == X_P_FULL || i == X_S_EMPTY) ? (uint32_t)kRowThreads : 1u);
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
    } else if (threadIdx.x == 32) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_r);
    }
    if (warp == 1) ptx::tmem_alloc(bar0 + 8u * 32u, 512);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t *>(sh.ptr + p.off_bar + 8 * 32), 0);
    // TMEM columns: S at 0, T at 128, O at 384; P at 448 (d = 64) or over S (d = 128)
    constexpr uint32_t tS = 0, tT = 128, tO = 384, tP = P_OWN ? 448 : 0;

    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };

    if (warp == 0) {
        // ---------------- loads
        bool ok = true;
        int issued = 0;
        if (J > 0) {
            ptx::mbar_expect_tx_w(bar(X_Q), (uint32_t)BM * D * 2);
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
                ptx::tma_load_3d_w(sh.base + p.off_q + (uint32_t)(h * BM * 128), &tm_q, bar(X_Q), 64 * h, i0, bh);
        }
        for (int j = 0; j < J && ok; ++j) {
            const int s = j % p.stages;
            const uint32_t round = (uint32_t)(j / p.stages);
            if (!(ok = wait_w(bar(X_KV_EMPTY + s), (round & 1u) ^ 1u))) break;
            const uint32_t fb = bar(X_KV_FULL + s);
            ptx::mbar_expect_tx_w(fb, (uint32_t)(2 * BN + kWin) * D * 2);
            const int j0 = j * BN;
            const int r0 = j0 - i0 - (BM - 1) + p.n - 1;  // table row of the window's first offset
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                ptx::tma_load_3d_w(sh.base + p.off_k + (uint32_t)s * p.stage_kv + (uint32_t)(h * BN * 128), &tm_k, fb,
                                   64 * h, j0, bh);
                ptx::tma_load_3d_w(sh.base + p.off_v + (uint32_t)s * p.stage_kv + (uint32_t)(h * BN * 128), &tm_v, fb,
                                   64 * h, j0, bh);
                ptx::tma_load_3d_w(sh.base + p.off_r + (uint32_t)s * p.stage_r + (uint32_t)(h * kWin * 128), &tm_r, fb,
                                   64 * h, r0, th);
            }
            issued = j + 1;
        }
        if (J > 0) tc::drain_bar(bar(X_Q), 0, sh.limit);
        for (int j = issued > p.stages ? issued - p.stages : 0; j < issued; ++j)
            tc::drain_bar(bar(X_KV_FULL + j % p.stages), (uint32_t)(j / p.stages) & 1u, sh.limit);
    } else if (warp == 1) {
        // ---------------- MMA issue
        bool ok = J > 0 ? wait_w(bar(X_Q), 0) : true;
        const uint64_t dq = ptx::sdesc_sw128(sh.base + p.off_q, 16, 1024);
        constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0);
        constexpr uint32_t idT = ptx::idesc_bf16(BM, kWin, 0);
        constexpr uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
        // S_j = Q K_j^T and T_j = Q R_win,j^T into their columns (free: the rows have read the
        // previous tile's S and T, and with P over S the previous P V is done)
        auto scores = [&](int j) -> bool {
            const int s = j % p.stages;
            if (!wait_w(bar(X_KV_FULL + s), (uint32_t)(j / p.stages) & 1u)) return false;
            if (j > 0 && !wait_w(bar(X_S_EMPTY), (uint32_t)(j - 1) & 1u)) return false;
            if (!P_OWN && j > 0 && !wait_w(bar(X_PV_DONE), (uint32_t)(j - 1) & 1u)) return false;
            ptx::tc_fence_after();
            const uint64_t dk = ptx::sdesc_sw128(sh.base + p.off_k + (uint32_t)s * p.stage_kv, 16, 1024);
            const uint64_t dr = ptx::sdesc_sw128(sh.base + p.off_r + (uint32_t)s * p.stage_r, 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::tc_mma_w(tmem + tS, dq + kstep(kk, BM), dk + kstep(kk, BN), idS, kk > 0 ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::tc_mma_w(tmem + tT, dq + kstep(kk, BM), dr + kstep(kk, kWin), idT, kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(bar(X_S_FULL));
            return true;
        };
        if (ok && J > 0) ok = scores(0);
        for (int j = 0; j < J && ok; ++j) {
            if (P_OWN && j + 1 < J && !(ok = scores(j + 1))) break;
            const int s = j % p.stages;
            if (!(ok = wait_w(bar(X_P_FULL), (uint32_t)j & 1u))) break;
            ptx::tc_fence_after();
            const uint64_t dv = ptx::sdesc_sw128(sh.base + p.off_v + (uint32_t)s * p.stage_kv, BN * 128, 1024);
#pragma unroll 1
            for (int kk = 0; kk < BN / 16; ++kk)  // O += P V
                ptx::tc_mma_ts_w(tmem + tO, tmem + tP + (uint32_t)(kk * 8), dv + mnstep(kk), idPV,
                                 (j > 0 || kk > 0) ? 1u : 0u);
            ptx::tc_commit_w(bar(X_PV_DONE));
            ptx::tc_commit_w(bar(X_KV_EMPTY + s));
            if (!P_OWN && j + 1 < J && !(ok = scores(j + 1))) break;
        }
        ptx::tc_commit_w(bar(X_DRAIN));
        tc::drain_bar(bar(X_DRAIN), 0, sh.limit);
    } else if (warp >= kRowWarp0) {
        // ---------------- NG threads per query row (TMEM lane = row): group g takes chunks
        // CPT g .. CPT g + CPT - 1 (32 keys each) of every tile; the row maximum and the row sum
        // are combined through shared memory at a named barrier of the row threads (every row
        // thread reaches each one: its waits are bounded)
        const int g = (warp - kRowWarp0) >> 2;
        const int quarter = warp & 3;
        const int il = 32 * quarter + lane, ii = i0 + il;
        const int tid = g * BM + il;  // 0 .. kRowThreads - 1
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        float *skew = reinterpret_cast<float *>(sh.ptr + p.off_skew) + tid * kSkew;
        float *ukb = reinterpret_cast<float *>(sh.ptr + p.off_uk);   // [2][BN]
        float *vrb = reinterpret_cast<float *>(sh.ptr + p.off_vr);   // [2][kWin]
        float *uv = reinterpret_cast<float *>(sh.ptr + p.off_uv);    // u [D], then v [D]
        float *X = reinterpret_cast<float *>(sh.ptr + p.off_x);      // [NG][BM]: the groups' values
        for (int e = tid; e < 2 * D; e += kRowThreads)
            uv[e] = __bfloat162float(e < D ? p.u[(long long)th * D + e] : p.vb[(long long)th * D + e - D]);
        ptx::named_bar_sync(1, kRowThreads);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < J && ok; ++j) {
            ok = tc::wait_bar(bar(X_S_FULL), (uint32_t)j & 1u, sh, p.err);
            ok = __all_sync(0xffffffffu, ok) != 0;
            const int s = j % p.stages, j0 = j * BN;
            // terms (c) and (d) of this tile: u.k for its 128 keys, v.r for its 256 offsets; two
            // buffers by tile parity
            float *uk = ukb + (j & 1) * BN;
            float *vr = vrb + (j & 1) * kWin;
            if (ok) {
                ptx::tc_fence_after();
                const uint8_t *kt = sh.ptr + p.off_k + s * p.stage_kv;
                const uint8_t *rt = sh.ptr + p.off_r + s * p.stage_r;
                if (g == 0) uk[il] = swz_dot<D>(kt, BN * 128, il, uv);
                for (int o = tid; o < kWin; o += kRowThreads) vr[o] = swz_dot<D>(rt, kWin * 128, o, uv + D);
            }
            if (!(ok = ptx::bar_red_and(1, kRowThreads, ok))) break;
            // pass 1: this group's logits (log2 domain), kept in registers, and their maximum
            float x[32 * CPT];
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                const int ch = CPT * g + cc;
                float sv[32], ta[32], tb[32];
                const int cb = 32 * (ch - quarter + 3);  // first T column the warp's rows need
                ptx::tmem_ld32f(lane_base + tS + (uint32_t)(32 * ch), sv);
                ptx::tmem_ld32f(lane_base + tT + (uint32_t)cb, ta);
                ptx::tmem_ld32f(lane_base + tT + (uint32_t)(cb + 32), tb);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    reinterpret_cast<float4 *>(skew)[q4] =
                        make_float4(ta[4 * q4] + vr[cb + 4 * q4], ta[4 * q4 + 1] + vr[cb + 4 * q4 + 1],
                                    ta[4 * q4 + 2] + vr[cb + 4 * q4 + 2], ta[4 * q4 + 3] + vr[cb + 4 * q4 + 3]);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    reinterpret_cast<float4 *>(skew)[8 + q4] =
                        make_float4(tb[4 * q4] + vr[cb + 32 + 4 * q4], tb[4 * q4 + 1] + vr[cb + 33 + 4 * q4],
                                    tb[4 * q4 + 2] + vr[cb + 34 + 4 * q4], tb[4 * q4 + 3] + vr[cb + 35 + 4 * q4]);
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int jl = 32 * ch + t, jj = j0 + jl;
                    const bool valid = ii < p.n && jj < nk && (!p.causal || jj <= ii);
                    const float tv = skew[t - lane + 31];  // column (j - i) + 127 of T, plus v.r
                    const float xv = valid ? p.c * (sv[t] + tv + uk[jl]) : -INFINITY;
                    mx = fmaxf(mx, xv);
                    x[32 * cc + t] = xv;
                }
            }
            // S and T are read: the next tile's products may overwrite them
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_S_EMPTY));
            // O and (with its own columns) P hold the previous tile's product until its P V is
            // done; the barrier below carries the outcome of this wait to every row thread
            if (j > 0) {
                ok = tc::wait_bar(bar(X_PV_DONE), (uint32_t)(j - 1) & 1u, sh, p.err);
                ok = __all_sync(0xffffffffu, ok) != 0;
                ptx::tc_fence_after();
            }
            X[tid] = mx;
            if (!(ok = ptx::bar_red_and(1, kRowThreads, ok))) break;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) mx = fmaxf(mx, X[gg * BM + il]);
            // lazy rescale: only when the maximum grows by more than 2^8
            const bool grow = mx > -INFINITY && (m == -INFINITY || mx > m + kRescaleLog2);
            const float m_new = grow ? fmaxf(m, mx) : m;
            const float al = grow ? ptx::ex2(m - m_new) : 1.f;  // m = -inf: 0 (nothing summed yet)
            if (j > 0 && __any_sync(0xffffffffu, grow && al != 1.f)) {  // this group's O columns
#pragma unroll 1
                for (int c0 = 32 * g; c0 < D; c0 += 32 * NG) {
                    float o[32];
                    ptx::tmem_ld32f(lane_base + tO + (uint32_t)c0, o);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] *= al;
                    __syncwarp();
                    ptx::tmem_st32f(lane_base + tO + (uint32_t)c0, o);
                }
                ptx::tmem_st_wait();
            }
            l *= al;
            m = m_new;
            // pass 2: P (bf16) for this group's keys
            {
#pragma unroll
                for (int cc = 0; cc < CPT; ++cc) {
                    const int ch = CPT * g + cc;
                    uint32_t pp[16];
#pragma unroll
                    for (int t2 = 0; t2 < 16; ++t2) {
                        const float a0 = x[32 * cc + 2 * t2], a1 = x[32 * cc + 2 * t2 + 1];
                        const float p0 = a0 == -INFINITY ? 0.f : ptx::ex2(a0 - m);
                        const float p1 = a1 == -INFINITY ? 0.f : ptx::ex2(a1 - m);
                        l += p0 + p1;
                        pp[t2] = ptx::pack_bf16x2(p0, p1);
                    }
                    __syncwarp();
                    ptx::tmem_st16(lane_base + tP + (uint32_t)(16 * ch), pp);
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_P_FULL));
        }
        // epilogue: the groups' row sums, then O / l -> bf16, group g writing the 32-column
        // blocks g, g + NG, ...
        float *XL = X + NG * BM;  // row sums apart from the maxima, which a slower thread may still read
        XL[tid] = l;
        ok = ptx::bar_red_and(1, kRowThreads, ok);
        if (ok && J > 0) {
            ok = tc::wait_bar(bar(X_PV_DONE), (uint32_t)(J - 1) & 1u, sh, p.err);
            ok = __all_sync(0xffffffffu, ok) != 0;
            if (ok) ptx::tc_fence_after();
        }
        if (ok) {
            float lt = 0.f;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) lt += XL[gg * BM + il];
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            uint4 *orow = reinterpret_cast<uint4 *>(p.out + ((long long)bh * p.n + ii) * D);
#pragma unroll 1
            for (int c0 = 32 * g; c0 < D; c0 += 32 * NG) {
                float o[32];
                if (J > 0) {
                    ptx::tmem_ld32f(lane_base + tO + (uint32_t)c0, o);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] = 0.f;
                }
                if (ii < p.n) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        orow[c0 / 8 + q] = make_uint4(ptx::pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                                                      ptx::pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                                      ptx::pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                                      ptx::pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
                }
            }
        }
    }
    ptx::tc_fence_before();
    ptx::cta_barrier();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch(const TxlArgs &a, cudaStream_t s) {
    const tc::DeviceInfo di = tc::device_info();
    if (di.sms <= 0 || di.smem_optin <= 0) return cudaErrorInvalidDevice;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.BH = a.B * a.H;
    p.H = a.H;
    p.n = a.n;
    p.n_tiles = (a.n + BM - 1) / BM;
    p.causal = a.causal;
    p.shared = a.shared;
    p.c = a.scale * kLog2e;
    p.kv_len = a.kv_len;
    p.err = a.err;
    p.u = static_cast<const __nv_bfloat16 *>(a.u);
    p.vb = static_cast<const __nv_bfloat16 *>(a.vb);
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.wait_limit = a.wait_limit > 0 ? a.wait_limit : 2000000000ll;
    if (p.BH == 0 || a.n == 0) return cudaSuccess;
    if ((long long)p.BH * p.n_tiles > INT32_MAX) return cudaErrorNotSupported;
    // shared memory: Q, the K / V / R_win rings (TMA targets, 1024-aligned), the diagonal
    // scratch, u.k and v.r (two tiles each), u and v, barriers
    auto layout = [&](int stages) {
        uint32_t off = 0;
        p.stage_kv = (uint32_t)BN * D * 2;
        p.stage_r = (uint32_t)kWin * D * 2;
        p.off_q = off; off += (uint32_t)BM * D * 2;
        p.off_k = off; off += (uint32_t)stages * p.stage_kv;
        p.off_v = off; off += (uint32_t)stages * p.stage_kv;
        p.off_r = off; off += (uint32_t)stages * p.stage_r;
        p.off_skew = off; off += (uint32_t)Groups<D>::kRowThreads * kSkew * 4;
        p.off_uk = off; off += 2 * BN * 4;
        p.off_vr = off; off += 2 * kWin * 4;
        p.off_uv = off; off += 2 * D * 4;
        p.off_x = off; off += 2u * Groups<D>::NG * BM * 4;
        p.off_bar = off; off += 8 * 32 + 16;
        p.stages = stages;
        return off + 1024;
    };
    uint32_t smem = layout(2);
    if (smem > (uint32_t)di.smem_optin) smem = layout(1);
    if (smem > (uint32_t)di.smem_optin) return cudaErrorNotSupported;

    CUtensorMap tm[4];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    const uint64_t rows = 2 * n - 1, Ht = a.shared ? 1 : (uint64_t)a.H;
    if (!tc::make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !tc::make_map(&tm[1], a.k, d, n, BH, rs, hs, BN) ||
        !tc::make_map(&tm[2], a.v, d, n, BH, rs, hs, BN) ||
        !tc::make_map(&tm[3], a.rel, d, rows, Ht, rs, rows * d * 2, kWin))
        return cudaErrorInvalidValue;

    static std::mutex mu;
    static bool opted[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opted[dev]) {
            e = cudaFuncSetAttribute(txl_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin);
            if (e != cudaSuccess) return e;
            opted[dev] = true;
        }
    }
    txl_tc_kernel<D><<<(unsigned)(p.BH * p.n_tiles), Groups<D>::kThreads, smem, s>>>(tm[0], tm[1], tm[2], tm[3], p);
    return cudaGetLastError();
}

}  // namespace txltc

bool txl_tc_covers(const TxlArgs &a) { return a.bf16 && (a.d == 64 || a.d == 128); }

cudaError_t launch_txl_tc(const TxlArgs &a, cudaStream_t s) {
    if (!txl_tc_covers(a)) return cudaErrorNotSupported;
    return a.d == 64 ? txltc::launch<64>(a, s) : txltc::launch<128>(a, s);
}

}  // namespace relattn
