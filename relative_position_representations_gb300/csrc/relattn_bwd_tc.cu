// Gradients of the Shaw relation-aware attention forward on the tensor cores (bf16 inputs,
// head dimension 64 or 128, fp32 gradients).
//
// The pages state only the forward pass ("Self-Attention with Relative Position
// Representations" page, section 3.4: eq. 3, eq. 4 and the softmax); the gradients are the
// chain rule through it, with r = r_ij = clip(j - i, k) + k and c = scale * log2(e):
//   x_ij  = c (q_i . k_j + R_ir),            R = Q W^K^T          (log2-domain logit)
//   p_ij  = 2^(x_ij - lse_i),                 lse_i = log2 sum_j 2^x_ij
//   dp_ij = dz_i . v_j + Rv_ir,               Rv = dZ W^V^T
//   ds_ij = p_ij (dp_ij - D_i),               D_i = sum_j p_ij dp_ij
//   dq_i  = scale (sum_j ds_ij k_j + sum_r gamma_ir w^K_r),   dk_j = scale sum_i ds_ij q_i,
//   dv_j  = sum_i p_ij dz_i,   dw^K_r = scale sum_i gamma_ir q_i,   dw^V_r = sum_i beta_ir dz_i,
// with the bins beta_ir = sum_{j: r_ij = r} p_ij and gamma_ir = sum_{j: r_ij = r} ds_ij.
//
// Three kernels, in stream order:
//   stats   one CTA per (head, 128-row query tile): R and Rv by MMA, then S_j = Q K_j^T and
//           dP_j = dZ V_j^T per key tile (tcgen05, fp32 in TMEM) and an online softmax over
//           the tile's keys that yields lse_i, D_i and the two end bins (offsets at or
//           beyond -k and +k, rescaled sums). Per row it writes R'_ir = c R_ir - lse_i and
//           Rv'_ir = Rv_ir - D_i (so that the next kernel needs no other row statistic).
//   keys    one CTA per (head, 128-key tile), looping over the query tiles that see it:
//           S^T = K Q_i^T and dP^T = V dZ_i^T (lanes = keys), then per element
//           p = 2^(c s + R'[r]) and ds = p (dp + Rv'[r]); P^T (bf16) goes back into TMEM and
//           dS (bf16) into shared memory, and three more MMAs follow: dV += P^T dZ_i,
//           dK += dS^T Q_i (both accumulated in TMEM over the query tiles) and
//           dQ_i = dS K (added into dq with vector atomics). An interior bin (-k < j - i < k)
//           holds exactly one key of its row, so the thread of that key stores its p and ds
//           as the bin (the 32 lanes of a warp store consecutive bins of one row).
//   tables  one CTA per (head, query tile): the bins as bf16 tiles, then dq_i += scale
//           sum_r gamma_ir w^K_r, dW^K += scale Gamma^T Q and dW^V += Beta^T dZ on tcgen05
//           (the table gradients by vector atomic adds).
// No n x n or n x n x d tensor reaches memory; the workspace holds per-row values only.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "relattn_internal.h"
#include "relattn_tc_launch.cuh"

namespace relattn {
namespace btc {

using tc::BM;
using tc::BN;
using tc::kLog2e;
using tc::Shared;

constexpr int kThreads = 192;   // warp 0 loads, warp 1 issues MMAs, warps 2-5 one row each
constexpr int kKeysThreads = 320;  // stats and keys kernels: warps 2-9, two threads per row / key
constexpr int kRowWarp0 = 2;
constexpr int kMaxW = 128;      // staged table rows (k + 1 causal, 2k + 1 otherwise)
constexpr int kRec = 8;         // floats per row record
constexpr int kMaxStages = 2;

// row record: lse, D, then beta and gamma of the two end bins
enum : int { kRecLse = 0, kRecD = 1, kRecBL = 2, kRecGL = 3, kRecBR = 4, kRecGR = 5 };

struct Params {
    int B, H, n, BH, n_tiles;
    int clip_k, causal, W, Wp;   // staged rows W, rounded up to 16 (N of R = Q W^K^T)
    int ak, av, bins;            // tables present; bins = ak || av
    int SK, SV;                  // row strides (floats) of R' and Rv' in the workspace
    int SRk, SRv;                // row strides (floats) of the R and Rv rows in shared memory
    int table_heads;
    float c, scale;
    const int *kv_len;
    int *err;
    float *dq, *dk, *dv;
    float *ws_rk, *ws_rv, *ws_bb, *ws_gg, *ws_rec;  // ws_bb, ws_gg: interior bins [row][W]
    uint32_t off_q, off_dz, off_k, off_v, off_wk, off_wv, off_r, off_rv, off_ds, off_bar;
    uint32_t off_p, off_gb;      // one-tile kernel: the P tile and the gamma|beta tile
    uint32_t off_x;              // one-tile kernel: per-row values exchanged by the two halves
    uint32_t stage_bytes;        // stats: one K (or V) stage; keys: one Q/dZ/R'/Rv' stage
    int stages;
    long long wait_limit;
    float *daK, *daV;            // one-tile kernel: the table gradients (atomic adds)
    long long ths;               // their head stride (elements; 0 = one table)
};

__device__ __forceinline__ int keys_of(const Params &p, int bh) {
    return p.kv_len ? max(0, min(p.kv_len[bh / p.H], p.n)) : p.n;
}

// K-major operand with 128-byte swizzle, k-step kk of 16: 64-column block kk / 4 (rows x 128
// bytes apart), 32 bytes per step inside the block (descriptor units of 16 bytes)
__device__ __forceinline__ uint64_t kstep(int kk, int rows) {
    return (uint64_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
}
// MN-major operand with 128-byte swizzle, k-step kk of 16 rows: 16 x 128 bytes
__device__ __forceinline__ uint64_t mnstep(int kk) { return (uint64_t)(kk * 16 * 128 >> 4); }

// instruction descriptor, kind::f16 with A MN-major as well (bit 15)
__host__ __device__ constexpr uint32_t idesc_amn(uint32_t M, uint32_t N) {
    return ptx::idesc_bf16(M, N, 1) | (1u << 15);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}\n"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void red_add_v4(float *dst, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

struct Smem {
    Shared sh;
    uint32_t bar0;
    uint32_t tmem_slot;
};

__device__ __forceinline__ Smem setup_smem(uint8_t *smem_raw, const Params &p) {
    Smem s;
    const uint32_t raw = ptx::smem_u32(smem_raw);
    s.sh.base = (raw + 1023u) & ~1023u;
    s.sh.ptr = smem_raw + (s.sh.base - raw);
    s.bar0 = s.sh.base + p.off_bar;
    s.tmem_slot = s.bar0 + 8u * 32u;
    s.sh.abort_flag = reinterpret_cast<volatile int *>(s.sh.ptr + p.off_bar + 8 * 32 + 4);
    s.sh.limit = p.wait_limit;
    return s;
}

// ============================================================================ stats kernel
enum : int {
    A_LD0 = 0, A_R_FULL, A_R_EMPTY, A_S_FULL, A_S_EMPTY, A_DRAIN,
    A_KV_FULL = 6, A_KV_EMPTY = A_KV_FULL + kMaxStages, kABars = A_KV_EMPTY + kMaxStages
};

template <int D>
__global__ void __launch_bounds__(kKeysThreads, 1)
    bwd_stats_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dz,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_wk, const __grid_constant__ CUtensorMap tm_wv,
                     const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = setup_smem(smem_raw, p);
    const Shared &sh = sm.sh;
    auto bar = [&](int i) { return sm.bar0 + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // causal: longest rows first
    const int qt = p.n_tiles - 1 - (int)blockIdx.x / p.BH, bh = (int)blockIdx.x % p.BH;
    const int i0 = qt * BM;
    const int nk = keys_of(p, bh);
    const int nkc = p.causal ? min(nk, i0 + BM) : nk;
    const int J = (nkc + BN - 1) / BN;
    const int th = p.table_heads ? bh % p.H : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kABars; ++i)
            ptx::mbar_init(bar(i), (i == A_R_EMPTY || i == A_S_EMPTY) ? 256u : 1u);
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
    } else if (threadIdx.x == 32) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_dz);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        if (p.ak) ptx::tma_prefetch_desc(&tm_wk);
        if (p.av) ptx::tma_prefetch_desc(&tm_wv);
    }
    if (warp == 1) ptx::tmem_alloc(sm.tmem_slot, 256);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t *>(sh.ptr + p.off_bar + 8 * 32), 0);

    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };

    if (warp == 0) {
        // ---------------- loads: Q, dZ and the table rows, then the K/V ring
        bool ok = true;
        uint32_t bytes = 2u * BM * D * 2;
        if (p.ak) bytes += (uint32_t)p.Wp * D * 2;
        if (p.av) bytes += (uint32_t)p.Wp * D * 2;
        ptx::mbar_expect_tx_w(bar(A_LD0), bytes);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
            ptx::tma_load_3d_w(sh.base + p.off_q + (uint32_t)(h * BM * 128), &tm_q, bar(A_LD0), 64 * h, i0, bh);
            ptx::tma_load_3d_w(sh.base + p.off_dz + (uint32_t)(h * BM * 128), &tm_dz, bar(A_LD0), 64 * h, i0, bh);
            if (p.ak)
                ptx::tma_load_3d_w(sh.base + p.off_wk + (uint32_t)(h * p.Wp * 128), &tm_wk, bar(A_LD0), 64 * h, 0, th);
            if (p.av)
                ptx::tma_load_3d_w(sh.base + p.off_wv + (uint32_t)(h * p.Wp * 128), &tm_wv, bar(A_LD0), 64 * h, 0, th);
        }
        int issued = 0;
        for (int j = 0; j < J && ok; ++j) {
            const int s = j % p.stages;
            const uint32_t round = (uint32_t)(j / p.stages);
            if (!(ok = wait_w(bar(A_KV_EMPTY + s), (round & 1u) ^ 1u))) break;
            ptx::mbar_expect_tx_w(bar(A_KV_FULL + s), 2u * BN * D * 2);
            const uint32_t ks = sh.base + p.off_k + (uint32_t)s * p.stage_bytes;
            const uint32_t vs = sh.base + p.off_v + (uint32_t)s * p.stage_bytes;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                ptx::tma_load_3d_w(ks + (uint32_t)(h * BN * 128), &tm_k, bar(A_KV_FULL + s), 64 * h, j * BN, bh);
                ptx::tma_load_3d_w(vs + (uint32_t)(h * BN * 128), &tm_v, bar(A_KV_FULL + s), 64 * h, j * BN, bh);
            }
            issued = j + 1;
        }
        // drain: no copy may still be in flight when the CTA exits
        tc::drain_bar(bar(A_LD0), 0, sh.limit);
        for (int j = issued > p.stages ? issued - p.stages : 0; j < issued; ++j)
            tc::drain_bar(bar(A_KV_FULL + j % p.stages), (uint32_t)(j / p.stages) & 1u, sh.limit);
    } else if (warp == 1) {
        // ---------------- MMA issue
        const uint64_t dq = ptx::sdesc_sw128(sh.base + p.off_q, 16, 1024);
        const uint64_t ddz = ptx::sdesc_sw128(sh.base + p.off_dz, 16, 1024);
        bool ok = wait_w(bar(A_LD0), 0);
        if (ok) {
            ptx::tc_fence_after();
            const uint32_t idR = ptx::idesc_bf16(BM, (uint32_t)p.Wp, 0);
            if (p.ak) {
                const uint64_t dw = ptx::sdesc_sw128(sh.base + p.off_wk, 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::tc_mma_w(tmem, dq + kstep(kk, BM), dw + kstep(kk, p.Wp), idR, kk > 0 ? 1u : 0u);
            }
            if (p.av) {
                const uint64_t dw = ptx::sdesc_sw128(sh.base + p.off_wv, 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::tc_mma_w(tmem + 128, ddz + kstep(kk, BM), dw + kstep(kk, p.Wp), idR, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit_w(bar(A_R_FULL));
            ok = wait_w(bar(A_R_EMPTY), 0);
        }
        constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0);
        for (int j = 0; j < J && ok; ++j) {
            const int s = j % p.stages;
            const uint32_t round = (uint32_t)(j / p.stages);
            if (!(ok = wait_w(bar(A_KV_FULL + s), round & 1u))) break;
            if (j > 0 && !(ok = wait_w(bar(A_S_EMPTY), (uint32_t)(j - 1) & 1u))) break;
            ptx::tc_fence_after();
            const uint64_t dk = ptx::sdesc_sw128(sh.base + p.off_k + (uint32_t)s * p.stage_bytes, 16, 1024);
            const uint64_t dv = ptx::sdesc_sw128(sh.base + p.off_v + (uint32_t)s * p.stage_bytes, 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::tc_mma_w(tmem, dq + kstep(kk, BM), dk + kstep(kk, BN), idS, kk > 0 ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::tc_mma_w(tmem + 128, ddz + kstep(kk, BM), dv + kstep(kk, BN), idS, kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(bar(A_S_FULL));
            ptx::tc_commit_w(bar(A_KV_EMPTY + s));
        }
        ptx::tc_commit_w(bar(A_DRAIN));
        tc::drain_bar(bar(A_DRAIN), 0, sh.limit);
    } else if (warp >= kRowWarp0) {
        // ---------------- two threads per query row (TMEM lane = row): group g takes chunks
        // 2 g and 2 g + 1 (32 keys each) of every key tile and runs its own online softmax over
        // them; the halves' maxima, sums and end bins are combined once, at the end
        const int g = (warp - kRowWarp0) >> 2;
        const int quarter = warp & 3;
        const int il = 32 * quarter + lane, i = i0 + il;
        const bool row_ok = i < p.n;
        const long long row = (long long)bh * p.n + i;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        float *Rs = reinterpret_cast<float *>(sh.ptr + p.off_r) + il * p.SRk;
        float *Rvs = reinterpret_cast<float *>(sh.ptr + p.off_rv) + il * p.SRv;
        float *X = reinterpret_cast<float *>(sh.ptr + p.off_x);  // [value][group][row]
        auto xv = [&](int v, int gg) -> float & { return X[(v * 2 + gg) * BM + il]; };
        const int k = p.clip_k, W = p.W;
        const bool bidir = !p.causal;
        const int khi = p.causal ? 0 : k;  // largest offset with a staged row
        bool ok = tc::wait_bar(bar(A_R_FULL), 0, sh, p.err);
        ok = __all_sync(0xffffffffu, ok) != 0;
        if (ok) {  // group 0 reads R, group 1 Rv
            ptx::tc_fence_after();
            if (g == 0 ? p.ak : p.av) {
                for (int c0 = 0; c0 < p.Wp; c0 += 16) {
                    float x[16];
                    ptx::tmem_ld16p(lane_base + (g == 0 ? 0u : 128u) + (uint32_t)c0, reinterpret_cast<uint32_t *>(x));
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if (c0 + t < W) (g == 0 ? Rs : Rvs)[c0 + t] = x[t];
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(A_R_EMPTY));
        }
        // the R and Rv rows are visible to both halves; every row thread gets here (its wait is
        // bounded) and the AND of the outcome sends all of them on or out together
        ok = ptx::bar_red_and(1, 256, ok);
        float m = -INFINITY, l = 0.f, Dacc = 0.f, Lb = 0.f, Ld = 0.f, Rb = 0.f, Rd = 0.f;
        for (int j = 0; j < J && ok; ++j) {
            ok = tc::wait_bar(bar(A_S_FULL), (uint32_t)j & 1u, sh, p.err);
            if (!(ok = __all_sync(0xffffffffu, ok) != 0)) break;
            ptx::tc_fence_after();
            const int j0 = j * BN;
            // pass 1: logits (log2 domain) back over the scores, and their maximum
            float mx = -INFINITY;
#pragma unroll 1
            for (int ch = 2 * g; ch < 2 * g + 2; ++ch) {
                float s[32];
                ptx::tmem_ld32f(lane_base + (uint32_t)(32 * ch), s);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int jj = j0 + 32 * ch + t, dl = jj - i;
                    const bool valid = jj < nk && (!p.causal || dl <= 0);
                    const int r = min(max(dl, -k), khi) + k;
                    const float x = valid ? p.c * (s[t] + (p.ak ? Rs[r] : 0.f)) : -INFINITY;
                    mx = fmaxf(mx, x);
                    s[t] = x;
                }
                __syncwarp();
                ptx::tmem_st32f(lane_base + (uint32_t)(32 * ch), s);
            }
            ptx::tmem_st_wait();
            if (mx > -INFINITY) {
                const float mn = fmaxf(m, mx);
                const float al = ptx::ex2(m - mn);  // m = -inf: 0 (the sums are still 0)
                l *= al; Dacc *= al; Lb *= al; Ld *= al; Rb *= al; Rd *= al;
                m = mn;
            }
            {
                // pass 2: probabilities (unnormalised), D and the end bins. Every lane runs it
                // (the TMEM loads are warp-collective); a row with no allowed key so far has only
                // -inf logits, whose terms are 0
                const float mm = m == -INFINITY ? 0.f : m;
#pragma unroll 1
                for (int ch = 2 * g; ch < 2 * g + 2; ++ch) {
                    float x[32], dp[32];
                    ptx::tmem_ld32f(lane_base + (uint32_t)(32 * ch), x);
                    ptx::tmem_ld32f(lane_base + 128u + (uint32_t)(32 * ch), dp);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int jj = j0 + 32 * ch + t, dl = jj - i;
                        const int r = min(max(dl, -k), khi) + k;
                        const float pt = ptx::ex2(x[t] - mm);  // -inf logits: 0
                        const float dpf = dp[t] + (p.av ? Rvs[r] : 0.f);
                        const float tt = pt * dpf;
                        l += pt;
                        Dacc += tt;
                        // the end bins (every key at or beyond -k, or +k); the interior
                        // bins, one key each, are written by the keys kernel
                        const bool isL = r == 0, isR = bidir && r == 2 * k && !isL;
                        Lb += isL ? pt : 0.f;
                        Ld += isL ? tt : 0.f;
                        Rb += isR ? pt : 0.f;
                        Rd += isR ? tt : 0.f;
                    }
                    __syncwarp();
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(A_S_EMPTY));
        }
        // the two halves' running values, combined at their common maximum
        xv(0, g) = m; xv(1, g) = l; xv(2, g) = Dacc; xv(3, g) = Lb; xv(4, g) = Ld; xv(5, g) = Rb; xv(6, g) = Rd;
        ok = ptx::bar_red_and(1, 256, ok);
        // per row (group 0): lse, D and the end bins; R' = c R - lse and Rv' = Rv - D in place
        // over the shared-memory rows, then copied out by whole rows (coalesced)
        if (ok && row_ok && g == 0) {
            const float m0 = xv(0, 0), m1 = xv(0, 1);
            const float mt = fmaxf(m0, m1);
            const float a0 = m0 == -INFINITY ? 0.f : ptx::ex2(m0 - mt);
            const float a1 = m1 == -INFINITY ? 0.f : ptx::ex2(m1 - mt);
            auto comb = [&](int v) { return a0 * xv(v, 0) + a1 * xv(v, 1); };
            const float lt = comb(1);
            const float lse = lt > 0.f ? mt + __log2f(lt) : INFINITY;
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const float Dv = comb(2) * inv;
            const float bl = comb(3) * inv, br = comb(5) * inv;
            float4 *rec = reinterpret_cast<float4 *>(p.ws_rec + row * kRec);
            rec[0] = make_float4(lse, Dv, bl, comb(4) * inv - Dv * bl);
            rec[1] = make_float4(br, comb(6) * inv - Dv * br, 0.f, 0.f);
            if (p.ak) {
                for (int r = 0; r < W; ++r) Rs[r] = p.c * Rs[r] - lse;
            } else {
                Rs[0] = -lse;
            }
            if (p.av) {
                for (int r = 0; r < W; ++r) Rvs[r] = Rvs[r] - Dv;
            } else {
                Rvs[0] = -Dv;
            }
        }
        // every row thread gets here (its waits are bounded), so the named barrier cannot hang
        if (ptx::bar_red_and(1, 256, ok)) {
            const int rows = min(BM, p.n - i0);
            const int wk = p.ak ? W : 1, wv = p.av ? W : 1;
            const float *Rs0 = reinterpret_cast<const float *>(sh.ptr + p.off_r);
            const float *Rvs0 = reinterpret_cast<const float *>(sh.ptr + p.off_rv);
            const long long row0 = (long long)bh * p.n + i0;
            for (int rr = warp - kRowWarp0; rr < rows; rr += 8) {
                float *dk = p.ws_rk + (row0 + rr) * p.SK;
                float *dv = p.ws_rv + (row0 + rr) * p.SV;
                for (int e = lane; e < p.SK; e += 32) dk[e] = e < wk ? Rs0[rr * p.SRk + e] : 0.f;
                for (int e = lane; e < p.SV; e += 32) dv[e] = e < wv ? Rvs0[rr * p.SRv + e] : 0.f;
            }
        }
    }
    ptx::tc_fence_before();
    ptx::cta_barrier();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

// ============================================================================= keys kernel
enum : int {
    B_KV = 0, B_S_FULL, B_P_FULL, B_DQ_FULL, B_DQ_EMPTY, B_MMA_DONE, B_DKV, B_DRAIN,
    B_Q_FULL = 8, B_Q_EMPTY = B_Q_FULL + kMaxStages, kBBars = B_Q_EMPTY + kMaxStages
};

// shared-memory layout of one query stage: Q tile, dZ tile, R' rows, Rv' rows
template <int D>
struct QStage {
    static constexpr uint32_t kTile = (uint32_t)BM * D * 2;
    static __device__ __forceinline__ uint32_t q(const Params &p, int s) { return p.off_q + (uint32_t)s * p.stage_bytes; }
    static __device__ __forceinline__ uint32_t dz(const Params &p, int s) { return q(p, s) + kTile; }
    static __device__ __forceinline__ uint32_t rk(const Params &p, int s) { return q(p, s) + 2 * kTile; }
    static __device__ __forceinline__ uint32_t rv(const Params &p, int s) {
        return rk(p, s) + (uint32_t)BM * p.SK * 4;
    }
};

template <int D>
__global__ void __launch_bounds__(kKeysThreads, 1)
    bwd_keys_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dz,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = setup_smem(smem_raw, p);
    const Shared &sh = sm.sh;
    auto bar = [&](int i) { return sm.bar0 + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // causal: the key tiles with the most query tiles first
    const int jt = (int)blockIdx.x / p.BH, bh = (int)blockIdx.x % p.BH;
    const int j0 = jt * BN;
    const int nk = keys_of(p, bh);
    const int qs = p.causal ? jt : 0;
    const int NQ = j0 < nk ? p.n_tiles - qs : 0;
    using QS = QStage<D>;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kBBars; ++i)
            ptx::mbar_init(bar(i), (i == B_P_FULL || i == B_DQ_EMPTY) ? 256u : 1u);
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
    } else if (threadIdx.x == 32) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_dz);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) ptx::tmem_alloc(sm.tmem_slot, 512);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t *>(sh.ptr + p.off_bar + 8 * 32), 0);
    // TMEM columns: S^T (then P^T) at 0, dP^T (then dQ) at 128, dK at 256, dV at 256 + D
    constexpr uint32_t tS = 0, tDP = 128, tDK = 256, tDV = 256 + D;

    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };

    if (warp == 0) {
        // ---------------- loads: K and V of this tile once, then Q, dZ, R', Rv' per query tile
        bool ok = true;
        int issued = 0;
        if (NQ > 0) {
            ptx::mbar_expect_tx_w(bar(B_KV), 2u * BN * D * 2);
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                ptx::tma_load_3d_w(sh.base + p.off_k + (uint32_t)(h * BN * 128), &tm_k, bar(B_KV), 64 * h, j0, bh);
                ptx::tma_load_3d_w(sh.base + p.off_v + (uint32_t)(h * BN * 128), &tm_v, bar(B_KV), 64 * h, j0, bh);
            }
        }
        for (int pi = 0; pi < NQ && ok; ++pi) {
            const int qt = qs + pi, i0 = qt * BM;
            const int s = pi % p.stages;
            const uint32_t round = (uint32_t)(pi / p.stages);
            if (!(ok = wait_w(bar(B_Q_EMPTY + s), (round & 1u) ^ 1u))) break;
            const int rows = min(BM, p.n - i0);
            const uint32_t rk_bytes = (uint32_t)rows * p.SK * 4, rv_bytes = (uint32_t)rows * p.SV * 4;
            ptx::mbar_expect_tx_w(bar(B_Q_FULL + s), 2u * BM * D * 2 + rk_bytes + rv_bytes);
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                ptx::tma_load_3d_w(sh.base + QS::q(p, s) + (uint32_t)(h * BM * 128), &tm_q, bar(B_Q_FULL + s),
                                   64 * h, i0, bh);
                ptx::tma_load_3d_w(sh.base + QS::dz(p, s) + (uint32_t)(h * BM * 128), &tm_dz, bar(B_Q_FULL + s),
                                   64 * h, i0, bh);
            }
            const long long row0 = (long long)bh * p.n + i0;
            bulk_load(sh.base + QS::rk(p, s), p.ws_rk + row0 * p.SK, rk_bytes, bar(B_Q_FULL + s));
            bulk_load(sh.base + QS::rv(p, s), p.ws_rv + row0 * p.SV, rv_bytes, bar(B_Q_FULL + s));
            issued = pi + 1;
        }
        if (NQ > 0) tc::drain_bar(bar(B_KV), 0, sh.limit);
        for (int pi = issued > p.stages ? issued - p.stages : 0; pi < issued; ++pi)
            tc::drain_bar(bar(B_Q_FULL + pi % p.stages), (uint32_t)(pi / p.stages) & 1u, sh.limit);
    } else if (warp == 1) {
        // ---------------- MMA issue
        bool ok = NQ > 0 ? wait_w(bar(B_KV), 0) : true;
        const uint64_t dk_k = ptx::sdesc_sw128(sh.base + p.off_k, 16, 1024);            // K, K-major
        const uint64_t dv_k = ptx::sdesc_sw128(sh.base + p.off_v, 16, 1024);            // V, K-major
        const uint64_t dk_mn = ptx::sdesc_sw128(sh.base + p.off_k, BN * 128, 1024);     // K, MN-major
        const uint64_t ds_k = ptx::sdesc_sw128(sh.base + p.off_ds, 16, 1024);           // dS^T, K-major
        const uint64_t ds_mn = ptx::sdesc_sw128(sh.base + p.off_ds, BN * 128, 1024);    // dS, MN-major
        constexpr uint32_t idS = ptx::idesc_bf16(BN, BM, 0);
        constexpr uint32_t idG = ptx::idesc_bf16(BN, D, 1);    // dV, dK: B MN-major
        constexpr uint32_t idQ = idesc_amn(BM, D);             // dQ: A and B MN-major
        for (int pi = 0; pi < NQ && ok; ++pi) {
            const int s = pi % p.stages;
            const uint32_t round = (uint32_t)(pi / p.stages);
            if (!(ok = wait_w(bar(B_Q_FULL + s), round & 1u))) break;
            if (pi > 0) {
                // the previous tile's P^T and dS are read, and its dQ is out of TMEM
                if (!(ok = wait_w(bar(B_MMA_DONE), (uint32_t)(pi - 1) & 1u))) break;
                if (!(ok = wait_w(bar(B_DQ_EMPTY), (uint32_t)(pi - 1) & 1u))) break;
            }
            ptx::tc_fence_after();
            const uint64_t dq_k = ptx::sdesc_sw128(sh.base + QS::q(p, s), 16, 1024);
            const uint64_t ddz_k = ptx::sdesc_sw128(sh.base + QS::dz(p, s), 16, 1024);
            const uint64_t dq_mn = ptx::sdesc_sw128(sh.base + QS::q(p, s), BM * 128, 1024);
            const uint64_t ddz_mn = ptx::sdesc_sw128(sh.base + QS::dz(p, s), BM * 128, 1024);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)  // S^T = K Q^T
                ptx::tc_mma_w(tmem + tS, dk_k + kstep(kk, BN), dq_k + kstep(kk, BM), idS, kk > 0 ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)  // dP^T = V dZ^T
                ptx::tc_mma_w(tmem + tDP, dv_k + kstep(kk, BN), ddz_k + kstep(kk, BM), idS, kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(bar(B_S_FULL));
            if (!(ok = wait_w(bar(B_P_FULL), (uint32_t)pi & 1u))) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int kk = 0; kk < BM / 16; ++kk)  // dV += P^T dZ (P^T bf16 pairs: 16 columns per 32-query chunk)
                ptx::tc_mma_ts_w(tmem + tDV, tmem + tS + (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8),
                                 ddz_mn + mnstep(kk), idG, (pi > 0 || kk > 0) ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < BM / 16; ++kk)  // dK += dS^T Q
                ptx::tc_mma_w(tmem + tDK, ds_k + kstep(kk, BN), dq_mn + mnstep(kk), idG,
                              (pi > 0 || kk > 0) ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < BN / 16; ++kk)  // dQ = dS K
                ptx::tc_mma_w(tmem + tDP, ds_mn + mnstep(kk), dk_mn + mnstep(kk), idQ, kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(bar(B_DQ_FULL));
            ptx::tc_commit_w(bar(B_Q_EMPTY + s));
            ptx::tc_commit_w(bar(B_MMA_DONE));
        }
        if (NQ > 0) ptx::tc_commit_w(bar(B_DKV));
        ptx::tc_commit_w(bar(B_DRAIN));
        tc::drain_bar(bar(B_DRAIN), 0, sh.limit);
    } else if (warp >= kRowWarp0) {
        // ---------------- two threads per key (TMEM lane = key) for P and dS, group g taking the
        // queries 64 g .. 64 g + 63 of each query tile (the elements are independent given R'
        // and Rv', so the halves need no exchange); per query row for dQ, group g taking
        // columns 32 g, 32 g + 64, ...
        const int g = (warp - kRowWarp0) >> 2;
        const int quarter = warp & 3;
        const int jl = 32 * quarter + lane, j = j0 + jl;
        const bool kvalid = j < nk;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        const int k = p.clip_k;
        const int khi = p.causal ? 0 : k;  // largest offset with a staged row
        uint8_t *ds_row = sh.ptr + p.off_ds + jl * 128;
        const uint32_t sw = (uint32_t)(jl & 7);
        bool ok = true;
        for (int pi = 0; pi < NQ && ok; ++pi) {
            const int qt = qs + pi, i0 = qt * BM;
            const int s = pi % p.stages;
            ok = tc::wait_bar(bar(B_S_FULL), (uint32_t)pi & 1u, sh, p.err);
            if (!(ok = __all_sync(0xffffffffu, ok) != 0)) break;
            ptx::tc_fence_after();
            const float *rk = reinterpret_cast<const float *>(sh.ptr + QS::rk(p, s));
            const float *rv = reinterpret_cast<const float *>(sh.ptr + QS::rv(p, s));
#pragma unroll 1
            for (int ch = 2 * g; ch < 2 * g + 2; ++ch) {
                float sv[32], dpv[32];
                ptx::tmem_ld32f(lane_base + tS + (uint32_t)(32 * ch), sv);
                ptx::tmem_ld32f(lane_base + tDP + (uint32_t)(32 * ch), dpv);
                ptx::tmem_ld_wait();
                uint32_t pp[16], dd[16];
                // do the warp's 32 keys and this chunk's 32 queries reach an interior bin
                // (|j - i| < k)? Then each element of one is stored, fp32, as the bin of row i
                const int dmax = j0 + 32 * quarter + 31 - (i0 + 32 * ch);
                const int dmin = j0 + 32 * quarter - (i0 + 32 * ch + 31);
                // interior offsets: -k < j - i < k, or -k < j - i <= 0 causal
                const int dhi = p.causal ? 1 : k;
                const bool band = p.bins && dmax > -k && dmin < dhi;
                const long long brow0 = ((long long)bh * p.n + i0 + 32 * ch) * p.W;
#pragma unroll
                for (int t2 = 0; t2 < 16; ++t2) {
                    float pe[2], de[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = 2 * t2 + h;
                        const int il = 32 * ch + t, i = i0 + il, dl = j - i;
                        const bool valid = kvalid && i < p.n && (!p.causal || dl <= 0);
                        const int r = min(max(dl, -k), khi) + k;
                        const float x = p.c * sv[t] + rk[il * p.SK + (p.ak ? r : 0)];
                        // rows beyond n hold stale R', Rv': select, never multiply by 0
                        const float pr = valid ? ptx::ex2(x) : 0.f;
                        const float dr = dpv[t] + rv[il * p.SV + (p.av ? r : 0)];
                        pe[h] = pr;
                        de[h] = valid ? pr * dr : 0.f;
                        if (band && valid && dl > -k && dl < dhi) {  // interior bin r of row i
                            p.ws_bb[brow0 + t * p.W + r] = pr;
                            p.ws_gg[brow0 + t * p.W + r] = de[h];
                        }
                    }
                    pp[t2] = ptx::pack_bf16x2(pe[0], pe[1]);
                    dd[t2] = ptx::pack_bf16x2(de[0], de[1]);
                }
                __syncwarp();
                // P^T of these 32 queries over the first 16 columns of their own S^T chunk, which
                // this thread has read (the other group's chunks may not be read yet)
                ptx::tmem_st16(lane_base + tS + (uint32_t)(32 * ch), pp);
                // dS^T row jl, queries 32 ch .. 32 ch + 31: 128-byte swizzled rows, two 64-query blocks
                const uint32_t blk = (uint32_t)(ch >> 1) * (BN * 128);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t u = (uint32_t)((ch & 1) * 4 + w);
                    *reinterpret_cast<uint4 *>(ds_row + blk + ((u ^ sw) << 4)) =
                        make_uint4(dd[4 * w], dd[4 * w + 1], dd[4 * w + 2], dd[4 * w + 3]);
                }
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_P_FULL));
            // dQ rows (TMEM lane = query row of the tile)
            ok = tc::wait_bar(bar(B_DQ_FULL), (uint32_t)pi & 1u, sh, p.err);
            if (!(ok = __all_sync(0xffffffffu, ok) != 0)) break;
            ptx::tc_fence_after();
            const int qi = i0 + jl;
            float *dqr = p.dq + ((long long)bh * p.n + qi) * D;
#pragma unroll 1
            for (int c0 = 32 * g; c0 < D; c0 += 64) {
                float v[32];
                ptx::tmem_ld32f(lane_base + tDP + (uint32_t)c0, v);
                ptx::tmem_ld_wait();
                if (qi < p.n) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        red_add_v4(dqr + c0 + 4 * u, p.scale * v[4 * u], p.scale * v[4 * u + 1],
                                   p.scale * v[4 * u + 2], p.scale * v[4 * u + 3]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_DQ_EMPTY));
        }
        // dK and dV of this key tile
        if (ok && NQ > 0) {
            ok = tc::wait_bar(bar(B_DKV), 0, sh, p.err);
            ok = __all_sync(0xffffffffu, ok) != 0;
            if (ok) ptx::tc_fence_after();
        }
        if (ok) {
            const long long krow = (long long)bh * p.n + j;
#pragma unroll 1
            for (int c0 = 32 * g; c0 < D; c0 += 64) {
                float a[32], b[32];
                if (NQ > 0) {
                    ptx::tmem_ld32f(lane_base + tDK + (uint32_t)c0, a);
                    ptx::tmem_ld32f(lane_base + tDV + (uint32_t)c0, b);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) a[t] = b[t] = 0.f;
                }
                if (j < p.n) {
                    float4 *dkr = reinterpret_cast<float4 *>(p.dk + krow * D + c0);
                    float4 *dvr = reinterpret_cast<float4 *>(p.dv + krow * D + c0);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        dkr[u] = make_float4(p.scale * a[4 * u], p.scale * a[4 * u + 1], p.scale * a[4 * u + 2],
                                             p.scale * a[4 * u + 3]);
                        dvr[u] = make_float4(b[4 * u], b[4 * u + 1], b[4 * u + 2], b[4 * u + 3]);
                    }
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

// =========================================================================== tables kernel
// One CTA per (head, query tile). The row threads build the tile's bins as bf16 MMA operands,
// gamma and beta [BM rows][128 table rows] (two 64-column blocks, 128-byte swizzle, zero beyond
// W): the end bins from the stats kernel's records, the interior bins from the keys kernel.
// Then three MMAs:
//   dQ_tab = Gamma W^K      (M = rows, K = table rows, N = D; added into dq times scale)
//   dW^K  += Gamma^T Q      (M = table rows, K = rows; A MN-major over the same tile)
//   dW^V  += Beta^T dZ
// and the tile's share of the table gradients goes out by vector atomic adds.
enum : int { C_LD = 0, C_G_FULL, C_MMA_DONE, C_DRAIN, kCBars };

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tables_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dz,
                      const __grid_constant__ CUtensorMap tm_wk, const __grid_constant__ Params p,
                      float *daK, float *daV, long long ths) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = setup_smem(smem_raw, p);
    const Shared &sh = sm.sh;
    auto bar = [&](int i) { return sm.bar0 + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = (int)blockIdx.x / p.BH, bh = (int)blockIdx.x % p.BH;
    const int i0 = qt * BM, h = bh % p.H;
    const int th = p.table_heads ? h : 0;
    const long long tho = p.table_heads ? (long long)h * ths : 0;
    const int W = p.W, k = p.clip_k;
    const int rows = min(BM, p.n - i0);
    const long long row0 = (long long)bh * p.n + i0;
    constexpr uint32_t kCols = D == 64 ? 256u : 512u;  // dQ_tab, dW^K, dW^V: D columns each

    if (threadIdx.x == 0) {
        for (int i = 0; i < kCBars; ++i) ptx::mbar_init(bar(i), i == C_G_FULL ? 128u : 1u);
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
    } else if (threadIdx.x == 32) {
        if (p.ak) ptx::tma_prefetch_desc(&tm_q);
        if (p.ak) ptx::tma_prefetch_desc(&tm_wk);
        if (p.av) ptx::tma_prefetch_desc(&tm_dz);
    }
    if (warp == 1) ptx::tmem_alloc(sm.tmem_slot, kCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t *>(sh.ptr + p.off_bar + 8 * 32), 0);
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };

    if (warp == 0) {
        uint32_t bytes = 0;
        if (p.ak) bytes += (uint32_t)BM * D * 2 + (uint32_t)p.Wp * D * 2;
        if (p.av) bytes += (uint32_t)BM * D * 2;
        ptx::mbar_expect_tx_w(bar(C_LD), bytes);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
            if (p.ak) {
                ptx::tma_load_3d_w(sh.base + p.off_q + (uint32_t)(hh * BM * 128), &tm_q, bar(C_LD), 64 * hh, i0, bh);
                ptx::tma_load_3d_w(sh.base + p.off_wk + (uint32_t)(hh * p.Wp * 128), &tm_wk, bar(C_LD), 64 * hh, 0, th);
            }
            if (p.av)
                ptx::tma_load_3d_w(sh.base + p.off_dz + (uint32_t)(hh * BM * 128), &tm_dz, bar(C_LD), 64 * hh, i0, bh);
        }
        tc::drain_bar(bar(C_LD), 0, sh.limit);
    } else if (warp == 1) {
        bool ok = wait_w(bar(C_LD), 0) && wait_w(bar(C_G_FULL), 0);
        if (ok) {
            ptx::tc_fence_after();
            constexpr uint32_t idT = ptx::idesc_bf16(BM, D, 1);  // A K-major, B MN-major
            constexpr uint32_t idW = idesc_amn(BM, D);           // A and B MN-major
            if (p.ak) {
                const uint64_t dg_k = ptx::sdesc_sw128(sh.base + p.off_k, 16, 1024);
                const uint64_t dg_mn = ptx::sdesc_sw128(sh.base + p.off_k, BM * 128, 1024);
                const uint64_t dwk = ptx::sdesc_sw128(sh.base + p.off_wk, (uint32_t)p.Wp * 128, 1024);
                const uint64_t dq_mn = ptx::sdesc_sw128(sh.base + p.off_q, BM * 128, 1024);
#pragma unroll 1
                for (int kk = 0; kk < p.Wp / 16; ++kk)  // dQ_tab = Gamma W^K
                    ptx::tc_mma_w(tmem, dg_k + kstep(kk, BM), dwk + mnstep(kk), idT, kk > 0 ? 1u : 0u);
#pragma unroll 1
                for (int kk = 0; kk < BM / 16; ++kk)  // dW^K = Gamma^T Q
                    ptx::tc_mma_w(tmem + D, dg_mn + mnstep(kk), dq_mn + mnstep(kk), idW, kk > 0 ? 1u : 0u);
            }
            if (p.av) {
                const uint64_t db_mn = ptx::sdesc_sw128(sh.base + p.off_v, BM * 128, 1024);
                const uint64_t ddz_mn = ptx::sdesc_sw128(sh.base + p.off_dz, BM * 128, 1024);
#pragma unroll 1
                for (int kk = 0; kk < BM / 16; ++kk)  // dW^V = Beta^T dZ
                    ptx::tc_mma_w(tmem + 2 * D, db_mn + mnstep(kk), ddz_mn + mnstep(kk), idW, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit_w(bar(C_MMA_DONE));
        }
        ptx::tc_commit_w(bar(C_DRAIN));
        tc::drain_bar(bar(C_DRAIN), 0, sh.limit);
    } else if (warp >= kRowWarp0) {
        const int quarter = warp & 3;
        const int il = 32 * quarter + lane, i = i0 + il;
        const long long row = row0 + il;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        const int nk = keys_of(p, bh);
        // this row's bins, bf16, 8 table rows per 16-byte chunk
        float4 e0 = make_float4(0.f, 0.f, 0.f, 0.f), e1 = e0;
        bool live = false;
        if (il < rows) {
            const float4 *rec = reinterpret_cast<const float4 *>(p.ws_rec + row * kRec);
            e0 = rec[0];
            e1 = rec[1];
            live = e0.x < INFINITY;
        }
        uint8_t *grow = sh.ptr + p.off_k + il * 128;  // gamma tile (the keys area of the other kernels)
        uint8_t *brow = sh.ptr + p.off_v + il * 128;  // beta tile
        const uint32_t sw = (uint32_t)(il & 7);
        for (int c8 = 0; c8 < 16; ++c8) {
            uint32_t gp[4], bp[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float gv[2], bv[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = 8 * c8 + 2 * e + hh;
                    float bb = 0.f, gg = 0.f;
                    if (live && r < W) {
                        if (r == 0) {
                            bb = e0.z;
                            gg = e0.w;
                        } else if (!p.causal && r == 2 * k) {
                            bb = e1.x;
                            gg = e1.y;
                        } else {
                            const int jj = i + r - k;  // the one key of an interior bin
                            if (jj >= 0 && jj < nk && (!p.causal || jj <= i)) {
                                bb = p.ws_bb[row * W + r];
                                gg = p.ws_gg[row * W + r];
                            }
                        }
                    }
                    gv[hh] = gg;
                    bv[hh] = bb;
                }
                gp[e] = ptx::pack_bf16x2(gv[0], gv[1]);
                bp[e] = ptx::pack_bf16x2(bv[0], bv[1]);
            }
            const uint32_t off = (uint32_t)(c8 >> 3) * (BM * 128) + ((((uint32_t)c8 & 7u) ^ sw) << 4);
            if (p.ak) *reinterpret_cast<uint4 *>(grow + off) = make_uint4(gp[0], gp[1], gp[2], gp[3]);
            if (p.av) *reinterpret_cast<uint4 *>(brow + off) = make_uint4(bp[0], bp[1], bp[2], bp[3]);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C_G_FULL));
        bool ok = tc::wait_bar(bar(C_MMA_DONE), 0, sh, p.err);
        ok = __all_sync(0xffffffffu, ok) != 0;
        if (ok) {
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32], wkv[32], wvv[32];
                if (p.ak) {
                    ptx::tmem_ld32f(lane_base + (uint32_t)c0, v);
                    ptx::tmem_ld32f(lane_base + (uint32_t)(D + c0), wkv);
                }
                if (p.av) ptx::tmem_ld32f(lane_base + (uint32_t)(2 * D + c0), wvv);
                ptx::tmem_ld_wait();
                if (p.ak && il < rows) {  // TMEM lane = row of the tile
                    float4 *dst = reinterpret_cast<float4 *>(p.dq + row * D + c0);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float4 t = dst[u];
                        t.x += p.scale * v[4 * u];
                        t.y += p.scale * v[4 * u + 1];
                        t.z += p.scale * v[4 * u + 2];
                        t.w += p.scale * v[4 * u + 3];
                        dst[u] = t;
                    }
                }
                if (il < W) {  // TMEM lane = table row
                    if (p.ak) {
                        float *dst = daK + tho + (long long)il * D + c0;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            red_add_v4(dst + 4 * u, p.scale * wkv[4 * u], p.scale * wkv[4 * u + 1],
                                       p.scale * wkv[4 * u + 2], p.scale * wkv[4 * u + 3]);
                    }
                    if (p.av) {
                        float *dst = daV + tho + (long long)il * D + c0;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            red_add_v4(dst + 4 * u, wvv[4 * u], wvv[4 * u + 1], wvv[4 * u + 2], wvv[4 * u + 3]);
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    ptx::cta_barrier();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kCols);
    }
}

// ================================================================== one-tile kernel
// Sequences of at most 128 keys (d = 64, at most 48 staged table rows): one query tile and
// one key tile per head, so one CTA does the whole head with no workspace and no atomics on
// dq, dk, dv. R = Q W^K^T, Rv = dZ W^V^T, S = Q K^T and dP = dZ V^T by MMA; the row threads
// take the exact row statistics in three passes over TMEM (maximum; row sum and D; then P,
// dS and the bins) and write P and dS (bf16) and the bins gamma | beta (bf16, one tile:
// gamma in table columns 0..63, beta in 64..127) into shared memory. Then
//   dV = P^T dZ, dK = dS^T Q     (A MN-major over the [query][key] tiles)
//   dQ = dS K + Gamma W^K        (A K-major)
//   [dW^K; dW^V] = [Gamma | Beta]^T [Q | dZ]   (one M = 128, N = 128 product; its two
//                                 off-diagonal blocks are not used)
// and the outputs leave TMEM by row (dq, dk, dv plain stores, the table rows by atomic adds).
enum : int { S_LD = 0, S_A_FULL, S_G_FULL, S_OUT_FULL, S_DRAIN, kSBars };
constexpr int kShortMaxW = 48;
constexpr int kShortThreads = 320;  // warp 0 loads, warp 1 MMAs, warps 2-9 two threads per row

__device__ __forceinline__ void st_bf16_tile(uint8_t *tile, int row, int col, float v) {
    // element (row, col) of a [128 rows][128 cols] bf16 tile in two 64-column blocks with the
    // 128-byte swizzle
    const uint32_t off = (uint32_t)(col >> 6) * (BM * 128) + (uint32_t)row * 128 +
                         ((((uint32_t)(col & 63) >> 3) ^ ((uint32_t)row & 7u)) << 4) + ((uint32_t)(col & 7) << 1);
    *reinterpret_cast<__nv_bfloat16 *>(tile + off) = __float2bfloat16_rn(v);
}

template <int D>
__global__ void __launch_bounds__(kShortThreads, 1)
    bwd_short_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_dz,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_wk, const __grid_constant__ CUtensorMap tm_wv,
                     const __grid_constant__ Params p) {
    static_assert(D == 64, "one-tile kernel: d = 64");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = setup_smem(smem_raw, p);
    const Shared &sh = sm.sh;
    auto bar = [&](int i) { return sm.bar0 + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = (int)blockIdx.x;
    const int nk = keys_of(p, bh);
    const int th = p.table_heads ? bh % p.H : 0;
    const long long tho = p.table_heads ? (long long)(bh % p.H) * p.ths : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSBars; ++i) ptx::mbar_init(bar(i), i == S_G_FULL ? 256u : 1u);
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
    } else if (threadIdx.x == 32) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_dz);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        if (p.ak) ptx::tma_prefetch_desc(&tm_wk);
        if (p.av) ptx::tma_prefetch_desc(&tm_wv);
    }
    if (warp == 1) ptx::tmem_alloc(sm.tmem_slot, 512);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t *>(sh.ptr + p.off_bar + 8 * 32), 0);
    // TMEM columns: S at 0 and dP at 128 (then dV at 0, dK at 64, dQ at 128), R at 256 and Rv
    // at 384 (then [dW^K | . ; . | dW^V] at 256)
    constexpr uint32_t tS = 0, tDP = 128, tR = 256, tRv = 384, tDV = 0, tDK = 64, tDQ = 128, tW = 256;
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };

    if (warp == 0) {
        uint32_t bytes = 4u * BM * D * 2;
        if (p.ak) bytes += (uint32_t)p.Wp * D * 2;
        if (p.av) bytes += (uint32_t)p.Wp * D * 2;
        ptx::mbar_expect_tx_w(bar(S_LD), bytes);
        ptx::tma_load_3d_w(sh.base + p.off_q, &tm_q, bar(S_LD), 0, 0, bh);
        ptx::tma_load_3d_w(sh.base + p.off_dz, &tm_dz, bar(S_LD), 0, 0, bh);
        ptx::tma_load_3d_w(sh.base + p.off_k, &tm_k, bar(S_LD), 0, 0, bh);
        ptx::tma_load_3d_w(sh.base + p.off_v, &tm_v, bar(S_LD), 0, 0, bh);
        if (p.ak) ptx::tma_load_3d_w(sh.base + p.off_wk, &tm_wk, bar(S_LD), 0, 0, th);
        if (p.av) ptx::tma_load_3d_w(sh.base + p.off_wv, &tm_wv, bar(S_LD), 0, 0, th);
        tc::drain_bar(bar(S_LD), 0, sh.limit);
    } else if (warp == 1) {
        bool ok = wait_w(bar(S_LD), 0);
        const uint64_t dq_k = ptx::sdesc_sw128(sh.base + p.off_q, 16, 1024);
        const uint64_t ddz_k = ptx::sdesc_sw128(sh.base + p.off_dz, 16, 1024);
        if (ok) {
            ptx::tc_fence_after();
            const uint32_t idR = ptx::idesc_bf16(BM, (uint32_t)p.Wp, 0);
            if (p.ak) {
                const uint64_t dw = ptx::sdesc_sw128(sh.base + p.off_wk, 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::tc_mma_w(tmem + tR, dq_k + kstep(kk, BM), dw + kstep(kk, p.Wp), idR, kk > 0 ? 1u : 0u);
            }
            if (p.av) {
                const uint64_t dw = ptx::sdesc_sw128(sh.base + p.off_wv, 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::tc_mma_w(tmem + tRv, ddz_k + kstep(kk, BM), dw + kstep(kk, p.Wp), idR, kk > 0 ? 1u : 0u);
            }
            constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0);
            const uint64_t dk_k = ptx::sdesc_sw128(sh.base + p.off_k, 16, 1024);
            const uint64_t dv_k = ptx::sdesc_sw128(sh.base + p.off_v, 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)  // S = Q K^T
                ptx::tc_mma_w(tmem + tS, dq_k + kstep(kk, BM), dk_k + kstep(kk, BN), idS, kk > 0 ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)  // dP = dZ V^T
                ptx::tc_mma_w(tmem + tDP, ddz_k + kstep(kk, BM), dv_k + kstep(kk, BN), idS, kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(bar(S_A_FULL));
            ok = wait_w(bar(S_G_FULL), 0);
        }
        if (ok) {
            ptx::tc_fence_after();
            constexpr uint32_t idA = idesc_amn(BM, D);       // A and B MN-major, N = D
            constexpr uint32_t idQ = ptx::idesc_bf16(BM, D, 1);  // A K-major, B MN-major
            constexpr uint32_t idW = idesc_amn(BM, 2 * D);   // [Gamma | Beta]^T [Q | dZ]
            const uint64_t dp_mn = ptx::sdesc_sw128(sh.base + p.off_p, BN * 128, 1024);
            const uint64_t ds_mn = ptx::sdesc_sw128(sh.base + p.off_ds, BN * 128, 1024);
            const uint64_t ds_k = ptx::sdesc_sw128(sh.base + p.off_ds, 16, 1024);
            const uint64_t dz_mn = ptx::sdesc_sw128(sh.base + p.off_dz, BM * 128, 1024);
            const uint64_t dq_mn = ptx::sdesc_sw128(sh.base + p.off_q, BM * 128, 1024);  // [Q | dZ]
            const uint64_t dk_mn = ptx::sdesc_sw128(sh.base + p.off_k, BN * 128, 1024);
            const uint64_t dgb_mn = ptx::sdesc_sw128(sh.base + p.off_gb, BM * 128, 1024);
            const uint64_t dg_k = ptx::sdesc_sw128(sh.base + p.off_gb, 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < BM / 16; ++kk)  // dV = P^T dZ
                ptx::tc_mma_w(tmem + tDV, dp_mn + mnstep(kk), dz_mn + mnstep(kk), idA, kk > 0 ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < BM / 16; ++kk)  // dK = dS^T Q
                ptx::tc_mma_w(tmem + tDK, ds_mn + mnstep(kk), dq_mn + mnstep(kk), idA, kk > 0 ? 1u : 0u);
#pragma unroll 1
            for (int kk = 0; kk < BN / 16; ++kk)  // dQ = dS K
                ptx::tc_mma_w(tmem + tDQ, ds_k + kstep(kk, BM), dk_mn + mnstep(kk), idQ, kk > 0 ? 1u : 0u);
            if (p.ak) {  // dQ += Gamma W^K
                const uint64_t dwk = ptx::sdesc_sw128(sh.base + p.off_wk, (uint32_t)p.Wp * 128, 1024);
#pragma unroll 1
                for (int kk = 0; kk < p.Wp / 16; ++kk)
                    ptx::tc_mma_w(tmem + tDQ, dg_k + kstep(kk, BM), dwk + mnstep(kk), idQ, 1u);
            }
            if (p.bins) {
#pragma unroll 1
                for (int kk = 0; kk < BM / 16; ++kk)  // [Gamma | Beta]^T [Q | dZ]
                    ptx::tc_mma_w(tmem + tW, dgb_mn + mnstep(kk), dq_mn + mnstep(kk), idW, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit_w(bar(S_OUT_FULL));
        }
        ptx::tc_commit_w(bar(S_DRAIN));
        tc::drain_bar(bar(S_DRAIN), 0, sh.limit);
    } else if (warp >= kRowWarp0) {
        // two threads per row: group g takes keys 64 g .. 64 g + 63 (chunks 2 g, 2 g + 1); the row
        // maximum, sum, D and end bins are combined through shared memory at a named barrier
        // of the 256 row threads (every row thread reaches each one: its waits are bounded)
        const int g = (warp - kRowWarp0) >> 2;
        const int quarter = warp & 3;
        const int il = 32 * quarter + lane;  // query row of S and dP, key row of dV and dK
        const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
        float *Rs = reinterpret_cast<float *>(sh.ptr + p.off_r) + il * p.SRk;
        float *Rvs = reinterpret_cast<float *>(sh.ptr + p.off_rv) + il * p.SRv;
        float *X = reinterpret_cast<float *>(sh.ptr + p.off_x);  // [value][group][row]
        auto xv = [&](int v, int gg) -> float & { return X[(v * 2 + gg) * BM + il]; };
        uint8_t *prow = sh.ptr + p.off_p + il * 128;
        uint8_t *dsrow = sh.ptr + p.off_ds + il * 128;
        uint8_t *gb = sh.ptr + p.off_gb;
        const uint32_t sw = (uint32_t)(il & 7);
        const int k = p.clip_k, W = p.W;
        const int khi = p.causal ? 0 : k;
        const bool bidir = !p.causal;
        const bool row_ok = il < p.n;
        // this row of the bins tile starts at zero (group g: block g)
        if (p.bins) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(gb + g * (BM * 128) + il * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        bool ok = tc::wait_bar(bar(S_A_FULL), 0, sh, p.err);
        ok = __all_sync(0xffffffffu, ok) != 0;
        if (ok && (g == 0 ? p.ak : p.av)) {  // group 0 reads R, group 1 Rv
            ptx::tc_fence_after();
            for (int c0 = 0; c0 < p.Wp; c0 += 16) {
                float x[16];
                ptx::tmem_ld16p(lane_base + (g == 0 ? tR : tRv) + (uint32_t)c0, reinterpret_cast<uint32_t *>(x));
                ptx::tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (c0 + t < W) (g == 0 ? Rs : Rvs)[c0 + t] = g == 0 ? p.c * x[t] : x[t];
            }
        }
        ok = ptx::bar_red_and(1, 256, ok);
        // pass 1: logits (log2 domain) over the scores, and the maximum of this half
        if (ok) {
            ptx::tc_fence_after();
            float m = -INFINITY;
#pragma unroll 1
            for (int ch = 2 * g; ch < 2 * g + 2; ++ch) {
                float sv[32];
                ptx::tmem_ld32f(lane_base + tS + (uint32_t)(32 * ch), sv);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int j = 32 * ch + t, dl = j - il;
                    const bool valid = row_ok && j < nk && (!p.causal || dl <= 0);
                    const int r = min(max(dl, -k), khi) + k;
                    const float x = valid ? fmaf(p.c, sv[t], p.ak ? Rs[r] : 0.f) : -INFINITY;
                    m = fmaxf(m, x);
                    sv[t] = x;
                }
                __syncwarp();
                ptx::tmem_st32f(lane_base + tS + (uint32_t)(32 * ch), sv);
            }
            ptx::tmem_st_wait();
            xv(0, g) = m;
        }
        ok = ptx::bar_red_and(1, 256, ok);
        // pass 2: row sum and D = sum_j p_ij dp_ij of this half. Every lane runs the TMEM loads
        // (they are warp-collective); a row without an allowed key has every logit at -inf, so
        // with its maximum taken as 0 all its terms are exactly 0
        const float m = ok ? fmaxf(xv(0, 0), xv(0, 1)) : 0.f;
        const float mm = m == -INFINITY ? 0.f : m;
        if (ok) {
            float l = 0.f, Dacc = 0.f;
#pragma unroll 1
            for (int ch = 2 * g; ch < 2 * g + 2; ++ch) {
                float x[32], dp[32];
                ptx::tmem_ld32f(lane_base + tS + (uint32_t)(32 * ch), x);
                ptx::tmem_ld32f(lane_base + tDP + (uint32_t)(32 * ch), dp);
                ptx::tmem_ld_wait();
                float l0 = 0.f, l1 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int t = 0; t < 32; t += 2) {
                    const int j = 32 * ch + t;
                    const int r0 = min(max(j - il, -k), khi) + k, r1 = min(max(j + 1 - il, -k), khi) + k;
                    const float p0 = ptx::ex2(x[t] - mm), p1 = ptx::ex2(x[t + 1] - mm);
                    l0 += p0;
                    l1 += p1;
                    d0 = fmaf(p0, dp[t] + (p.av ? Rvs[r0] : 0.f), d0);
                    d1 = fmaf(p1, dp[t + 1] + (p.av ? Rvs[r1] : 0.f), d1);
                }
                l += l0 + l1;
                Dacc += d0 + d1;
            }
            xv(1, g) = l;
            xv(2, g) = Dacc;
        }
        ok = ptx::bar_red_and(1, 256, ok);
        const float l = ok ? xv(1, 0) + xv(1, 1) : 0.f;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float Dv = ok ? (xv(2, 0) + xv(2, 1)) * inv : 0.f;
        // pass 3: P, dS (bf16 tiles, block g) and the bins of this half's keys
        if (ok) {
            float Lb = 0.f, Lg = 0.f, Rb = 0.f, Rg = 0.f;
#pragma unroll 1
            for (int ch = 2 * g; ch < 2 * g + 2; ++ch) {
                float x[32], dp[32];
                ptx::tmem_ld32f(lane_base + tS + (uint32_t)(32 * ch), x);
                ptx::tmem_ld32f(lane_base + tDP + (uint32_t)(32 * ch), dp);
                ptx::tmem_ld_wait();
                uint32_t pp[16], dd[16];
#pragma unroll
                for (int t2 = 0; t2 < 16; ++t2) {
                    float pe[2], de[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = 2 * t2 + h, j = 32 * ch + t, dl = j - il;
                        const int r = min(max(dl, -k), khi) + k;
                        const float pr = ptx::ex2(x[t] - mm) * inv;  // -inf logits: 0
                        const float ds = pr * (dp[t] + (p.av ? Rvs[r] : 0.f) - Dv);
                        pe[h] = pr;
                        de[h] = ds;
                        if (p.bins && pr > 0.f) {
                            const bool isL = r == 0, isR = bidir && r == 2 * k && !isL;
                            Lb += isL ? pr : 0.f;
                            Lg += isL ? ds : 0.f;
                            Rb += isR ? pr : 0.f;
                            Rg += isR ? ds : 0.f;
                            if (!isL && !isR) {  // an interior bin: this one key
                                st_bf16_tile(gb, il, r, ds);
                                st_bf16_tile(gb, il, 64 + r, pr);
                            }
                        }
                    }
                    pp[t2] = ptx::pack_bf16x2(pe[0], pe[1]);
                    dd[t2] = ptx::pack_bf16x2(de[0], de[1]);
                }
                const uint32_t blk = (uint32_t)(ch >> 1) * (BN * 128);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t u = (uint32_t)((ch & 1) * 4 + w);
                    *reinterpret_cast<uint4 *>(prow + blk + ((u ^ sw) << 4)) =
                        make_uint4(pp[4 * w], pp[4 * w + 1], pp[4 * w + 2], pp[4 * w + 3]);
                    *reinterpret_cast<uint4 *>(dsrow + blk + ((u ^ sw) << 4)) =
                        make_uint4(dd[4 * w], dd[4 * w + 1], dd[4 * w + 2], dd[4 * w + 3]);
                }
            }
            xv(3, g) = Lb;
            xv(4, g) = Lg;
            xv(5, g) = Rb;
            xv(6, g) = Rg;
        }
        ok = ptx::bar_red_and(1, 256, ok);
        if (ok && g == 0 && p.bins && l > 0.f) {  // the end bins, both halves
            st_bf16_tile(gb, il, 0, xv(4, 0) + xv(4, 1));
            st_bf16_tile(gb, il, 64, xv(3, 0) + xv(3, 1));
            if (bidir && k > 0) {
                st_bf16_tile(gb, il, 2 * k, xv(6, 0) + xv(6, 1));
                st_bf16_tile(gb, il, 64 + 2 * k, xv(5, 0) + xv(5, 1));
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(S_G_FULL));
        if (ok) {
            ok = tc::wait_bar(bar(S_OUT_FULL), 0, sh, p.err);
            ok = __all_sync(0xffffffffu, ok) != 0;
        }
        if (ok) {  // group g: columns 32 g .. 32 g + 31 of every output
            ptx::tc_fence_after();
            const long long row = (long long)bh * p.n + il;
            const int c0 = 32 * g;
            float a[32], b[32], q[32];
            ptx::tmem_ld32f(lane_base + tDV + (uint32_t)c0, a);
            ptx::tmem_ld32f(lane_base + tDK + (uint32_t)c0, b);
            ptx::tmem_ld32f(lane_base + tDQ + (uint32_t)c0, q);
            ptx::tmem_ld_wait();
            if (il < p.n) {
                float4 *dv = reinterpret_cast<float4 *>(p.dv + row * D + c0);
                float4 *dk = reinterpret_cast<float4 *>(p.dk + row * D + c0);
                float4 *dq = reinterpret_cast<float4 *>(p.dq + row * D + c0);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    dv[u] = make_float4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
                    dk[u] = make_float4(p.scale * b[4 * u], p.scale * b[4 * u + 1], p.scale * b[4 * u + 2],
                                        p.scale * b[4 * u + 3]);
                    dq[u] = make_float4(p.scale * q[4 * u], p.scale * q[4 * u + 1], p.scale * q[4 * u + 2],
                                        p.scale * q[4 * u + 3]);
                }
            }
            // lane il < 64 (quarters 0 and 1): dW^K row il in columns 0..63; lane 64 + r: dW^V row
            // r in columns 64..127. The TMEM loads run warp-uniformly; the atomics only for table
            // rows that exist.
            const bool kpart = quarter < 2;
            const int r = kpart ? il : il - 64;
            if (p.bins && (kpart ? p.ak : p.av)) {
                float *dst = (kpart ? p.daK : p.daV) + tho + (long long)r * D + c0;
                const float f = kpart ? p.scale : 1.f;
                float v[32];
                ptx::tmem_ld32f(lane_base + tW + (uint32_t)((kpart ? 0 : D) + c0), v);
                ptx::tmem_ld_wait();
                if (r < W) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        red_add_v4(dst + 4 * u, f * v[4 * u], f * v[4 * u + 1], f * v[4 * u + 2], f * v[4 * u + 3]);
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

// ==================================================================================== host

inline uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }
inline unsigned long long round_up_ull(unsigned long long x, unsigned long long a) { return (x + a - 1) / a * a; }

// workspace floats per row and layout (each array 256-byte aligned)
inline unsigned long long ws_layout(const BwdArgs &a, int W, int SK, int SV, Params *p) {
    const unsigned long long rows = (unsigned long long)a.B * a.H * a.n;
    unsigned long long off = 0;
    auto take = [&](unsigned long long floats) {
        const unsigned long long o = off;
        off = round_up_ull(off + floats * 4, 256);
        return o;
    };
    const unsigned long long o_rk = take(rows * SK), o_rv = take(rows * SV);
    const unsigned long long o_bb = take(rows * W), o_gg = take(rows * W), o_rec = take(rows * kRec);
    if (p) {
        char *b = static_cast<char *>(a.workspace);
        p->ws_rk = reinterpret_cast<float *>(b + o_rk);
        p->ws_rv = reinterpret_cast<float *>(b + o_rv);
        p->ws_bb = reinterpret_cast<float *>(b + o_bb);
        p->ws_gg = reinterpret_cast<float *>(b + o_gg);
        p->ws_rec = reinterpret_cast<float *>(b + o_rec);
    }
    return off;
}

template <typename K>
cudaError_t opt_in(K kern, std::mutex &mu, bool (&opted)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!opted[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::device_info().smem_optin);
        if (e != cudaSuccess) return e;
        opted[dev] = true;
    }
    return cudaSuccess;
}

// one-tile kernel: shared-memory layout (Q and dZ adjacent: [Q | dZ] is one operand),
// descriptors and launch
template <int D>
cudaError_t launch_short(const BwdArgs &a, Params p, cudaStream_t s) {
    const tc::DeviceInfo di = tc::device_info();
    const bool ak = a.aK != nullptr, av = a.aV != nullptr;
    const uint32_t tile = (uint32_t)BM * D * 2;
    const uint32_t tab = round_up((uint32_t)p.Wp * D * 2, 1024);
    uint32_t off = 0;
    p.off_q = off; off += tile;
    p.off_dz = off; off += tile;
    p.off_k = off; off += tile;
    p.off_v = off; off += tile;
    p.off_wk = off; if (ak) off += tab;
    p.off_wv = off; if (av) off += tab;
    p.off_p = off; off += (uint32_t)BM * BN * 2;
    p.off_ds = off; off += (uint32_t)BM * BN * 2;
    p.off_gb = off; off += (uint32_t)BM * 128 * 2;
    p.off_r = off; off += (uint32_t)BM * p.SRk * 4;
    p.off_rv = off; off += (uint32_t)BM * p.SRv * 4;
    off = round_up(off, 16);
    p.off_x = off; off += 7 * 2 * BM * 4;
    p.off_bar = off; off += 8 * 32 + 16;
    const uint32_t smem = off + 1024;
    if (smem > (uint32_t)di.smem_optin) return cudaErrorNotSupported;
    CUtensorMap tm[6];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    if (!tc::make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !tc::make_map(&tm[1], a.dout, d, n, BH, rs, hs, BM) ||
        !tc::make_map(&tm[2], a.k, d, n, BH, rs, hs, BN) || !tc::make_map(&tm[3], a.v, d, n, BH, rs, hs, BN))
        return cudaErrorInvalidValue;
    tm[4] = tm[0];
    tm[5] = tm[0];
    const uint64_t Ht = p.table_heads ? (uint64_t)a.H : 1;
    const uint64_t rows_mem = (uint64_t)(2 * a.clip_k + 1);
    const uint64_t ths_bytes = p.table_heads ? (uint64_t)a.ths * 2 : rows_mem * d * 2;
    if (ak && !tc::make_map(&tm[4], a.aK, d, rows_mem, Ht, rs, ths_bytes, (uint32_t)p.Wp)) return cudaErrorInvalidValue;
    if (av && !tc::make_map(&tm[5], a.aV, d, rows_mem, Ht, rs, ths_bytes, (uint32_t)p.Wp)) return cudaErrorInvalidValue;
    static std::mutex mu;
    static bool opted[64] = {};
    cudaError_t e;
    if ((e = opt_in(bwd_short_kernel<D>, mu, opted)) != cudaSuccess) return e;
    const int Htab = p.table_heads ? a.H : 1;
    const size_t tab_bytes = (size_t)((long long)(Htab - 1) * a.ths + (long long)(2 * a.clip_k + 1) * a.d) * sizeof(float);
    if (ak && (e = cudaMemsetAsync(a.daK, 0, tab_bytes, s)) != cudaSuccess) return e;
    if (av && (e = cudaMemsetAsync(a.daV, 0, tab_bytes, s)) != cudaSuccess) return e;
    bwd_short_kernel<D><<<(unsigned)p.BH, kShortThreads, smem, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch(const BwdArgs &a, cudaStream_t s) {
    const bool ak = a.aK != nullptr, av = a.aV != nullptr;
    const int W = a.causal ? a.clip_k + 1 : 2 * a.clip_k + 1;
    if ((ak || av) && W > kMaxW) return cudaErrorNotSupported;
    const tc::DeviceInfo di = tc::device_info();
    if (di.sms <= 0 || di.smem_optin <= 0) return cudaErrorInvalidDevice;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.B = a.B;
    p.H = a.H;
    p.n = a.n;
    p.BH = a.B * a.H;
    p.n_tiles = (a.n + BM - 1) / BM;
    p.clip_k = a.clip_k;
    p.causal = a.causal;
    p.W = W;
    p.Wp = (int)round_up((uint32_t)W, 16);
    p.ak = ak;
    p.av = av;
    p.bins = ak || av;
    p.SK = (int)round_up((uint32_t)(ak ? W : 1), 4);
    p.SV = (int)round_up((uint32_t)(av ? W : 1), 4);
    // even strides: the band gather of a warp's 32 rows (address step SR - 1) hits 32 banks;
    // without the table one slot holds the row's -lse (or -D)
    p.SRk = ak ? (W + 1) & ~1 : 2;
    p.SRv = av ? (W + 1) & ~1 : 2;
    p.table_heads = a.ths != 0 ? 1 : 0;
    p.c = a.scale * kLog2e;
    p.scale = a.scale;
    p.kv_len = a.kv_len;
    p.err = a.err;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.wait_limit = a.wait_limit > 0 ? a.wait_limit : 2000000000ll;
    if (p.BH == 0 || a.n == 0) return cudaSuccess;
    if ((long long)p.BH * p.n_tiles > INT32_MAX) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(a.workspace) % 256 != 0) return cudaErrorNotSupported;
    ws_layout(a, W, p.SK, p.SV, &p);
    p.daK = a.daK;
    p.daV = a.daV;
    p.ths = a.ths;
    if constexpr (D == 64) {
        if (a.n <= BM && (!(ak || av) || W <= kShortMaxW)) {
            const cudaError_t e = launch_short<D>(a, p, s);
            if (e != cudaErrorNotSupported) return e;
        }
    }

    // stats kernel shared memory: Q, dZ, K/V stages, table rows (TMA targets, 1024-aligned),
    // then the R and Rv rows and the barriers
    const uint32_t tile = (uint32_t)BM * D * 2;
    const uint32_t tab = (uint32_t)p.Wp * D * 2;
    auto layout_a = [&](Params &q, int stages) {
        uint32_t off = 0;
        q.off_q = off; off += tile;
        q.off_dz = off; off += tile;
        q.off_k = off; off += (uint32_t)stages * tile;
        q.off_v = off; off += (uint32_t)stages * tile;
        q.off_wk = off; if (ak) off += round_up(tab, 1024);
        q.off_wv = off; if (av) off += round_up(tab, 1024);
        q.off_r = off; off += (uint32_t)BM * q.SRk * 4;
        q.off_rv = off; off += (uint32_t)BM * q.SRv * 4;
        off = round_up(off, 16);
        q.off_x = off; off += 7 * 2 * BM * 4;
        q.off_bar = off; off += 8 * 32 + 16;
        q.stage_bytes = tile;
        q.stages = stages;
        return off + 1024;  // slack to align the base to 1024 bytes
    };
    // keys kernel shared memory: K, V, dS (MMA operands, 1024-aligned), the query stages
    // (Q, dZ, R' rows, Rv' rows), barriers
    auto layout_b = [&](Params &q, int stages) {
        uint32_t off = 0;
        q.off_k = off; off += tile;
        q.off_v = off; off += tile;
        q.off_ds = off; off += (uint32_t)BN * BM * 2;
        q.stage_bytes = round_up(2 * tile + (uint32_t)BM * (q.SK + q.SV) * 4, 1024);
        q.off_q = off; off += (uint32_t)stages * q.stage_bytes;
        q.off_bar = off; off += 8 * 32 + 16;
        q.stages = stages;
        return off + 1024;
    };
    const uint32_t optin = (uint32_t)di.smem_optin;
    Params pa = p, pb = p;
    // two K/V stages when there is more than one key tile and they fit
    uint32_t sma = layout_a(pa, p.n_tiles > 1 ? 2 : 1);
    if (sma > optin) sma = layout_a(pa, 1);
    uint32_t smb = layout_b(pb, 2);
    if (smb > optin) smb = layout_b(pb, 1);
    if (sma > optin || smb > optin) return cudaErrorNotSupported;
    // tables kernel shared memory: Q, dZ, W^K (TMA), the gamma and beta tiles (in the places
    // of the K and V tiles), barriers
    Params pc = p;
    auto layout_c = [&](Params &q) {
        uint32_t off = 0;
        q.off_q = off; off += tile;
        q.off_dz = off; off += tile;
        q.off_wk = off; off += round_up(tab, 1024);
        q.off_k = off; off += (uint32_t)BM * 128 * 2;   // gamma: 128 rows x 128 table rows, bf16
        q.off_v = off; off += (uint32_t)BM * 128 * 2;   // beta
        q.off_bar = off; off += 8 * 32 + 16;
        return off + 1024;
    };
    const uint32_t smc = layout_c(pc);
    if (smc > optin) return cudaErrorNotSupported;

    // TMA descriptors
    CUtensorMap tm[6];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    if (!tc::make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !tc::make_map(&tm[1], a.dout, d, n, BH, rs, hs, BM) ||
        !tc::make_map(&tm[2], a.k, d, n, BH, rs, hs, BN) || !tc::make_map(&tm[3], a.v, d, n, BH, rs, hs, BN))
        return cudaErrorInvalidValue;
    tm[4] = tm[0];
    tm[5] = tm[0];
    const uint64_t Ht = p.table_heads ? (uint64_t)a.H : 1;
    const uint64_t rows_mem = (uint64_t)(2 * a.clip_k + 1);
    const uint64_t ths_bytes = p.table_heads ? (uint64_t)a.ths * 2 : rows_mem * d * 2;
    if (ak && !tc::make_map(&tm[4], a.aK, d, rows_mem, Ht, rs, ths_bytes, (uint32_t)p.Wp)) return cudaErrorInvalidValue;
    if (av && !tc::make_map(&tm[5], a.aV, d, rows_mem, Ht, rs, ths_bytes, (uint32_t)p.Wp)) return cudaErrorInvalidValue;

    static std::mutex mu;
    static bool opted_a[64] = {}, opted_b[64] = {}, opted_c[64] = {};
    cudaError_t e;
    if ((e = opt_in(bwd_stats_kernel<D>, mu, opted_a)) != cudaSuccess) return e;
    if ((e = opt_in(bwd_keys_kernel<D>, mu, opted_b)) != cudaSuccess) return e;
    if ((e = opt_in(bwd_tables_kernel<D>, mu, opted_c)) != cudaSuccess) return e;

    const int Htab = p.table_heads ? a.H : 1;
    const size_t tab_bytes = (size_t)((long long)(Htab - 1) * a.ths + (long long)(2 * a.clip_k + 1) * a.d) * sizeof(float);
    if (ak && (e = cudaMemsetAsync(a.daK, 0, tab_bytes, s)) != cudaSuccess) return e;
    if (av && (e = cudaMemsetAsync(a.daV, 0, tab_bytes, s)) != cudaSuccess) return e;
    // dq: the keys kernel adds dS K into it, the tables kernel the table term
    if ((e = cudaMemsetAsync(a.dq, 0, (size_t)p.BH * a.n * D * sizeof(float), s)) != cudaSuccess) return e;
    const unsigned tiles = (unsigned)(p.BH * p.n_tiles);
    bwd_stats_kernel<D><<<tiles, kKeysThreads, sma, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], pa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_keys_kernel<D><<<tiles, kKeysThreads, smb, s>>>(tm[0], tm[1], tm[2], tm[3], pb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ak || av) {
        bwd_tables_kernel<D><<<tiles, kThreads, smc, s>>>(tm[0], tm[1], tm[4], pc, a.daK, a.daV, a.ths);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace btc

unsigned long long bwd_tc_workspace_bytes(int B, int H, int n, int clip_k) {
    BwdArgs a{};
    a.B = B;
    a.H = H;
    a.n = n;
    const int W = 2 * clip_k + 1;
    const int S4 = (int)btc::round_up((uint32_t)W, 4);
    return btc::ws_layout(a, W, S4, S4, nullptr);
}

bool bwd_tc_covers(const BwdArgs &a) {
    if (!a.bf16 || (a.d != 64 && a.d != 128)) return false;
    const int W = a.causal ? a.clip_k + 1 : 2 * a.clip_k + 1;
    if ((a.aK || a.aV) && W > btc::kMaxW) return false;
    return reinterpret_cast<uintptr_t>(a.workspace) % 256 == 0;
}

cudaError_t launch_bwd_tc(const BwdArgs &a, cudaStream_t s) {
    if (!bwd_tc_covers(a)) return cudaErrorNotSupported;
    return a.d == 64 ? btc::launch<64>(a, s) : btc::launch<128>(a, s);
}

}  // namespace relattn
