// Relation-aware attention forward for short sequences (at most 256 keys), bf16 in / fp32
// accumulate, head dimension 64, for sm_103a. The arithmetic is that of the long-sequence
// kernel ("Self-Attention with Relative Position Representations", section 3.4: eq. 4 split
// as in "Efficient Implementation", e_ij = scale (q_i . k_j + R_i[clip(j-i,k)+k]) with
// R = Q W^K^T, and eq. 3 as z_i = sum_j a_ij v_j + sum_r beta_ir w^V_r with
// beta_ir = sum_{j: clip(j-i,k)+k = r} a_ij); what differs is how the work is laid out.
//
// A unit is one query tile of 128 rows of one head with all of its keys (one or two key tiles
// of 128). Two CTAs share an SM, each running its units one after the other (CTA b takes
// units b, b + gridDim.x, ..., longest causal tiles first), so one CTA's softmax overlaps the
// other's loads and MMAs. A CTA holds 256 TMEM columns:
//   S  [0, 128)    the scores S_j = Q K_j^T; after the unit's last tile, the value bins (bf16)
//   P  [128, 192)  R = Q W^K^T (read out at the start of the unit), then P_j (bf16 pairs)
//   O  [192, 256)  the output accumulator
// Roles (256 threads):
//   warp 0      TMA loads: Q with W^K, the K ring, the V ring, W^V; the next unit's Q and K
//               are loaded as soon as this unit's score MMAs have read theirs.
//   warp 1      MMA issue (one elected lane): R and S_0 under one commit, S_1 once the
//               softmax has read S_0, then P_j V_j and beta W^V.
//   warps 2, 3  idle (registers are handed out per group of four warps).
//   warps 4-7   softmax and epilogue, one thread per query row (TMEM lane = row): the score
//               row is read half a tile (64 keys) at a time, twice: the first pass forms the
//               logits and the maximum (logits that are not kept raw go back over the scores),
//               the second the exponentials, P and the bins; the relative term is a per-row constant
//               on 32-key chunks beyond +-k (kept raw, folded into the exponent) and a
//               gather from R in shared memory inside the band; online softmax in the exp2
//               domain with a lazy rescale; value bins in shared memory; O / l -> bf16 into a
//               staging tile, stored by one bulk tensor copy.
// R and the bins sit in shared memory transposed ([table row][query row]), so every gather
// and every store of a warp touches 32 distinct banks.
// Every wait is bounded; a wait that runs out sets the device status word and the CTA drains
// and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "relattn_tc_kernel.cuh"

namespace relattn {
namespace sk {

using tc::BM;
using tc::BN;
using tc::KB;
using tc::NCH;
using tc::kLog2e;
using tc::kRescaleLog2;
using tc::Shared;

constexpr int D = 64;
constexpr int kThreads = 256;
constexpr int kSoftWarp0 = 4;
// registers per thread: launched with kLaunchRegs (two CTAs per SM fill the register file);
// the producer/MMA group hands registers to the softmax group
constexpr int kLaunchRegs = 128;
constexpr int kCtrlRegs = 56;
constexpr int kSoftRegs = 200;
static_assert(128 * kCtrlRegs + 128 * kSoftRegs == kThreads * kLaunchRegs, "register split");
constexpr int kMaxTiles = 2;     // key tiles per unit
constexpr int kMaxStages = 2;    // per K or V ring
constexpr int kTmemCols = 256;
constexpr int kMaxW = 64;        // staged table rows: R must fit the P columns
constexpr int kSoftBar = 1;      // hardware named barrier of the 128 softmax threads

struct Tm {
    static constexpr uint32_t S = 0, P = 128, O = 192;
};

enum : int {
    X_Q_FULL = 0, X_Q_EMPTY, X_AV_FULL, X_AV_EMPTY,
    X_S_FULL, X_S_EMPTY, X_P_FULL, X_PV_DONE, X_BN_FULL, X_O_FULL, X_O_EMPTY, X_DRAIN,
    X_K_FULL = 12,
    X_K_EMPTY = X_K_FULL + kMaxStages,
    X_V_FULL = X_K_EMPTY + kMaxStages,
    X_V_EMPTY = X_V_FULL + kMaxStages,
    kNumBars = X_V_EMPTY + kMaxStages
};

struct Params {
    int BH, H, n, n_qtiles, num_units;
    float scale_log2;         // scale * log2(e)
    const int *kv_len;        // [B] or null
    int *err;                 // device status word
    void *out;                // [B, H, n, 64] bf16
    int clip_k;               // k
    int W;                    // table rows used: k + 1 (causal) or 2k + 1
    int npad_k, kpad_v;       // W rounded up to 16: N of R = Q W^K^T, K of beta W^V
    int table_heads;          // 1: tables indexed by head, 0: one shared table
    uint32_t off_q, off_k, off_v, off_ak, off_av, off_r, off_bins, off_bar;
    uint32_t off_stage;       // the output tile (16 KB, 1024-aligned) over R and the bins
    int kstages, vstages;     // 1 or 2
    long long wait_limit;     // bound of every wait, SM clock cycles
    int withhold_q;           // test hook: the producer issues no Q load for its first unit
};

// a unit: head bh, query tile qt, allowed keys nk, keys the tile may see nkc, key tiles J
template <bool CAUSAL>
struct Unit {
    int bh, qt, nk, nkc, J;
    __device__ __forceinline__ void make(const Params &p, int t) {
        qt = p.n_qtiles - 1 - t / p.BH;
        bh = t - (p.n_qtiles - 1 - qt) * p.BH;
        nk = p.kv_len ? max(0, min(p.kv_len[bh / p.H], p.n)) : p.n;
        nkc = CAUSAL ? min(nk, qt * BM + BM) : nk;
        J = (nkc + BN - 1) / BN;
    }
};

// keys of tile j that are loaded and multiplied: the allowed keys in whole 32-key boxes
__device__ __forceinline__ int tile_cols(int nkc, int j) {
    const int c = nkc - j * BN;
    return c >= BN ? BN : ((c + KB - 1) / KB) * KB;
}

// ring entry e of a ring with 1 or 2 stages -> stage and round
__device__ __forceinline__ void ring(int stages, uint32_t e, uint32_t &st, uint32_t &round) {
    st = stages == 1 ? 0u : (e & 1u);
    round = stages == 1 ? e : (e >> 1);
}

__device__ __forceinline__ uint32_t bar_addr(const Shared &sh, const Params &p, int i) {
    return sh.base + p.off_bar + 8u * (uint32_t)i;
}

// ======================================================================= loads
template <bool AK, bool AV, bool CAUSAL>
__device__ void producer(const Params &p, const Shared &sh, const CUtensorMap *tm_q,
                         const CUtensorMap *tm_k, const CUtensorMap *tm_v, const CUtensorMap *tm_kf,
                         const CUtensorMap *tm_vf, const CUtensorMap *tm_ak, const CUtensorMap *tm_av) {
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    uint32_t q_it = 0, k_it = 0, v_it = 0, av_it = 0;
    bool ok = true;
    // K (isK) or V tile j of the unit into the next stage of its ring
    auto load_kv = [&](bool isK, const Unit<CAUSAL> &u, int j) -> bool {
        uint32_t &it = isK ? k_it : v_it;
        uint32_t st, round;
        ring(isK ? p.kstages : p.vstages, it, st, round);
        const uint32_t fb = bar((isK ? X_K_FULL : X_V_FULL) + (int)st);
        if (!wait(bar((isK ? X_K_EMPTY : X_V_EMPTY) + (int)st), (round & 1u) ^ 1u)) return false;
        const int nbox = tile_cols(u.nkc, j) / KB;
        ptx::mbar_expect_tx_w(fb, (uint32_t)nbox * KB * D * 2);
        const uint32_t dst = sh.base + (isK ? p.off_k : p.off_v) + st * (uint32_t)(BN * D * 2);
        if (nbox == BN / KB) {
            ptx::tma_load_3d_w(dst, isK ? tm_kf : tm_vf, fb, 0, j * BN, u.bh);
        } else {
            for (int b = 0; b < nbox; ++b)
                ptx::tma_load_3d_w(dst + (uint32_t)(b * KB * 128), isK ? tm_k : tm_v, fb, 0,
                                   j * BN + b * KB, u.bh);
        }
        ++it;
        return true;
    };
    for (int i = 0; ok; ++i) {
        const int t = (int)blockIdx.x + i * (int)gridDim.x;
        if (t >= p.num_units) break;
        Unit<CAUSAL> u;
        u.make(p, t);
        if (u.J == 0) continue;
        const int th = p.table_heads ? u.bh % p.H : 0;
        if (!(ok = wait(bar(X_Q_EMPTY), (q_it & 1u) ^ 1u))) break;
        ++q_it;
        ptx::mbar_expect_tx_w(bar(X_Q_FULL), (uint32_t)(BM + (AK ? p.npad_k : 0)) * D * 2);
        // test hook: the first unit's Q tile is announced but never loaded, so the MMA warp's
        // bounded wait for it runs out (the device status word reports the timeout)
        if (!(p.withhold_q && q_it == 1))
            ptx::tma_load_3d_w(sh.base + p.off_q, tm_q, bar(X_Q_FULL), 0, u.qt * BM, u.bh);
        if (AK) ptx::tma_load_3d_w(sh.base + p.off_ak, tm_ak, bar(X_Q_FULL), 0, 0, th);
        for (int j = 0; j < u.J && ok; ++j) ok = load_kv(true, u, j);
        for (int j = 0; j < u.J && ok; ++j) ok = load_kv(false, u, j);
        if (!ok) break;
        if (AV) {
            if (!(ok = wait(bar(X_AV_EMPTY), (av_it & 1u) ^ 1u))) break;
            ++av_it;
            ptx::mbar_expect_tx_w(bar(X_AV_FULL), (uint32_t)p.kpad_v * D * 2);
            ptx::tma_load_3d_w(sh.base + p.off_av, tm_av, bar(X_AV_FULL), 0, 0, th);
        }
    }
    // drain: wait (bounded) for the copies issued into shared memory, so that none is still
    // in flight when the CTA exits (normally all were consumed; after an abort the consumers
    // may have given up on some)
    for (int side = 0; side < 2; ++side) {
        const uint32_t it = side == 0 ? k_it : v_it;
        const int stages = side == 0 ? p.kstages : p.vstages;
        for (uint32_t e = it > (uint32_t)stages ? it - stages : 0u; e < it; ++e) {
            uint32_t st, round;
            ring(stages, e, st, round);
            tc::drain_bar(bar((side == 0 ? X_K_FULL : X_V_FULL) + (int)st), round & 1u, sh.limit);
        }
    }
    if (q_it) tc::drain_bar(bar(X_Q_FULL), (q_it - 1u) & 1u, sh.limit);
    if (AV && av_it) tc::drain_bar(bar(X_AV_FULL), (av_it - 1u) & 1u, sh.limit);
}

// ======================================================================= MMA issue
// The whole warp runs the role with warp-uniform control flow; one elected lane issues every
// tcgen05 instruction.
template <bool AK, bool AV, bool CAUSAL>
__device__ void mma(const Params &p, const Shared &sh, uint32_t tmem) {
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    constexpr uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
    constexpr uint32_t kStage = (uint32_t)(BN * D * 2);
    // K-major operands (Q, K, W^K): 128-byte rows, a k-step of 16 moves 32 bytes inside the
    // swizzle atom; MN-major operands (V, W^V): 16 rows of 128 bytes per k-step. The
    // descriptors are formed at each use (few registers stay live in this warp).
    auto kmaj = [&](uint32_t off) { return ptx::sdesc_sw128(sh.base + off, 16, 1024); };
    // one count per ring or barrier: S issues = K entries, P waits = V entries, bins = W^V loads
    uint32_t q_it = 0, k_it = 0, v_it = 0, av_it = 0, o_it = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
        const int t = (int)blockIdx.x + i * (int)gridDim.x;
        if (t >= p.num_units) break;
        Unit<CAUSAL> u;
        u.make(p, t);
        if (u.J == 0) continue;
        // every MMA of the previous unit is done: it read P and the bins from the columns
        // that R and S_0 are about to overwrite
        if (o_it && !(ok = wait(bar(X_O_FULL), (o_it - 1u) & 1u))) break;
        if (!(ok = wait(bar(X_Q_FULL), q_it & 1u))) break;
        ++q_it;
        ptx::tc_fence_after();
        if (AK)  // R = Q W^K^T into the P columns (one chain of four k-steps)
            ptx::tc_mma_ss_k64(tmem + Tm::P, kmaj(p.off_q), kmaj(p.off_ak),
                               ptx::idesc_bf16(BM, (uint32_t)p.npad_k, 0), 0u);
        for (int j = 0; j < u.J && ok; ++j) {  // S_j = Q K_j^T once the softmax has read S_{j-1}
            if (!(ok = wait(bar(X_S_EMPTY), (k_it & 1u) ^ 1u))) break;
            uint32_t st, round;
            ring(p.kstages, k_it, st, round);
            ++k_it;
            if (!(ok = wait(bar(X_K_FULL + (int)st), round & 1u))) break;
            ptx::tc_fence_after();
            ptx::tc_mma_ss_k64(tmem + Tm::S, kmaj(p.off_q), kmaj(p.off_k + st * kStage),
                               ptx::idesc_bf16(BM, (uint32_t)tile_cols(u.nkc, j), 0), 0u);
            ptx::tc_commit_w(bar(X_S_FULL));
            ptx::tc_commit_w(bar(X_K_EMPTY + (int)st));
            if (j == u.J - 1) ptx::tc_commit_w(bar(X_Q_EMPTY));  // Q and W^K are read
        }
        for (int j = 0; j < u.J && ok; ++j) {  // O (+)= P_j V_j
            if (!(ok = wait(bar(X_P_FULL), v_it & 1u))) break;
            uint32_t st, round;
            ring(p.vstages, v_it, st, round);
            ++v_it;
            if (!(ok = wait(bar(X_V_FULL + (int)st), round & 1u))) break;
            // the first product overwrites O: the previous unit's epilogue has read it
            if (j == 0 && !(ok = wait(bar(X_O_EMPTY), (o_it & 1u) ^ 1u))) break;
            ptx::tc_fence_after();
            const uint64_t dv = ptx::sdesc_sw128(sh.base + p.off_v + st * kStage, BN * 128, 1024);
            const int nk16 = tile_cols(u.nkc, j) / 16;
            if (nk16 == BN / 16) {  // a whole tile: one chain of eight k-steps
                ptx::tc_mma_ts_k128(tmem + Tm::O, tmem + Tm::P, dv, idPV, j > 0 ? 1u : 0u);
            } else {
#pragma unroll 1
                for (int kk = 0; kk < nk16; ++kk)
                    ptx::tc_mma_ts_w(tmem + Tm::O, tmem + Tm::P + (uint32_t)(kk * 8),
                                     dv + (uint64_t)(kk * 16 * 128 >> 4), idPV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::tc_commit_w(bar(X_PV_DONE));
            ptx::tc_commit_w(bar(X_V_EMPTY + (int)st));
        }
        if (!ok) break;
        if (AV) {  // O += beta W^V, beta (bf16 pairs) in the S columns
            if (!(ok = wait(bar(X_BN_FULL), av_it & 1u))) break;
            if (!(ok = wait(bar(X_AV_FULL), av_it & 1u))) break;
            ++av_it;
            ptx::tc_fence_after();
            const uint64_t dav = ptx::sdesc_sw128(sh.base + p.off_av, (uint32_t)p.kpad_v * 128, 1024);
#pragma unroll 1
            for (int kk = 0; kk < p.kpad_v / 16; ++kk)
                ptx::tc_mma_ts_w(tmem + Tm::O, tmem + Tm::S + (uint32_t)(kk * 8),
                                 dav + (uint64_t)(kk * 16 * 128 >> 4), idPV, 1u);
            ptx::tc_commit_w(bar(X_AV_EMPTY));
        }
        ptx::tc_commit_w(bar(X_O_FULL));
        ++o_it;
    }
    // every MMA issued by this warp completes before TMEM is released
    ptx::tc_commit_w(bar(X_DRAIN));
    tc::drain_bar(bar(X_DRAIN), 0, sh.limit);
}

// ======================================================================= softmax / epilogue
__device__ __forceinline__ float2 pair(const float *x, int e) { return make_float2(x[e], x[e + 1]); }
__device__ __forceinline__ void put(float *x, int e, float2 v) {
    x[e] = v.x;
    x[e + 1] = v.y;
}
__device__ __forceinline__ float2 dup(float v) { return make_float2(v, v); }

template <bool AK, bool AV, bool CAUSAL>
__device__ void softmax(const Params &p, const Shared &sh, uint32_t tmem, const CUtensorMap *tm_o) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stid = threadIdx.x - 32 * kSoftWarp0;  // 0 .. 127; thread 0 issues the tile stores
    auto uni = [](int v) { return __shfl_sync(0xffffffffu, v, 0); };
    const int quad = uni(warp & 3);  // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;
    const uint32_t lb = tmem + ((uint32_t)(quad * 32) << 16);
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    // column r of this row's R and bins: element r * BM (transposed layout)
    float *Rt = reinterpret_cast<float *>(sh.ptr + p.off_r) + row;
    float *Bt = reinterpret_cast<float *>(sh.ptr + p.off_bins) + row;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.f;  // raw chunks need max(x * sl2) = sl2 * max(x)
    const int k = p.clip_k, W = p.W;
    const int hi_lim = CAUSAL ? 0 : k;  // offsets at or beyond it take the last table row
    uint32_t s_it = 0, pv_it = 0, o_it = 0;
    bool ok = true;
    // Only the first warp polls an mbarrier; the other three meet it at the named barrier,
    // which carries the outcome (an AND over the 128 threads) to every thread.
    auto wait_w = [&](int b, uint32_t parity) -> bool {
        bool r = true;
        if (quad == 0) {
            r = tc::wait_bar(bar(b), parity, sh, p.err);
            r = __all_sync(0xffffffffu, r ? 1 : 0) != 0;
        }
        r = ptx::bar_red_and(kSoftBar, 128, r);
        ptx::tc_fence_after();
        __syncwarp();
        return r;
    };

    // the next unit is decoded (and its key length loaded) while the current one runs
    int t = (int)blockIdx.x;
    Unit<CAUSAL> nxt;
    if (t < p.num_units) nxt.make(p, t);
    while (t < p.num_units && ok) {
        const Unit<CAUSAL> u = nxt;
        const int bh = uni(u.bh), qt = uni(u.qt), nk = uni(u.nk), nkc = uni(u.nkc), J = uni(u.J);
        t += (int)gridDim.x;
        if (t < p.num_units) nxt.make(p, t);
        const int i0 = qt * BM, gi = i0 + row;
        const int gmin = uni(i0 + quad * 32), gmax = gmin + 31;  // rows of this warp
        if (J == 0) {  // no allowed key: the rows are zero
            if (gi < p.n) {
                __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) + ((long long)bh * p.n + gi) * D;
#pragma unroll
                for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4 *>(orow)[c] = make_uint4(0, 0, 0, 0);
            }
            continue;
        }
        // the previous tile store has read the staging tile, which R and the bins overlay; the
        // barrier in the wait below carries that to every thread
        if (stid == 0) ptx::bulk_wait_read0();
        if (!(ok = wait_w(X_S_FULL, s_it & 1u))) break;
        ++s_it;
        float c_left = 0.f, c_right = 0.f;  // relative term beyond the window on either side
        if (AK) {  // R row (scaled to the log2 domain) -> shared memory
#pragma unroll 1
            for (int c0 = 0; c0 < p.npad_k; c0 += 16) {
                uint32_t r[16];
                ptx::tmem_ld16(lb + Tm::P + (uint32_t)c0, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c0 + e < W) Rt[(c0 + e) * BM] = __uint_as_float(r[e]) * sl2;
            }
            c_left = Rt[0];
            c_right = Rt[(W - 1) * BM];
        }
        if (AV)
            for (int r = 0; r < W; ++r) Bt[r * BM] = 0.f;
        float m_ref = -INFINITY, l = 0.f, lsum = 0.f;

        for (int j = 0; j < J && ok; ++j) {
            const int j0 = j * BN;
            const int cols = tile_cols(nkc, j);  // multiple of 32, > 0
            int live = cols / KB;                // chunks any row of the warp sees
            if (CAUSAL) live = min(live, max(0, (gmax - j0) / KB + 1));
            if (j > 0) {
                if (!(ok = wait_w(X_S_FULL, s_it & 1u))) break;
                ++s_it;
            }
            // chunk c of the tile: its relative term is one constant for every row of the warp
            // (all offsets beyond the window on one side) and it needs no mask
            auto raw_chunk = [&](int c, float &cst) -> bool {
                const int e0 = j0 + c * KB;
                const bool w_left = (e0 + KB - 1 - gmin) <= -k;
                const bool w_right = (e0 - gmax) >= hi_lim;
                const bool full = (e0 + KB <= nk) && (!CAUSAL || e0 + KB - 1 <= gmin);
                cst = AK ? (w_left ? c_left : c_right) : 0.f;
                return (!AK || w_left || w_right) && full && pos_scale;
            };
            // ---- pass 1: logits in the log2 domain and the row maximum, half a tile at a
            // time; a chunk not kept raw gets its logits written back over its scores
            float rmax = -INFINITY;
#pragma unroll 1
            for (int hf = 0; hf < NCH / 2; ++hf) {
                if (2 * hf >= live) break;
                float x[2 * KB];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
                    if (2 * hf + cc < live) ptx::tmem_ld32f(lb + Tm::S + (uint32_t)((2 * hf + cc) * KB), x + cc * KB);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * hf + cc;
                    if (c >= live) continue;
                    float *xc = x + cc * KB;
                    float cst;
                    if (raw_chunk(c, cst)) {
                        rmax = fmaxf(rmax, fmaf(tc::max32(xc), sl2, cst));
                        continue;
                    }
                    const int e0 = j0 + c * KB;
                    const bool w_left = (e0 + KB - 1 - gmin) <= -k;
                    const bool w_right = (e0 - gmax) >= hi_lim;
                    const bool full = (e0 + KB <= nk) && (!CAUSAL || e0 + KB - 1 <= gmin);
                    if (!AK) {
#pragma unroll
                        for (int e = 0; e < KB; e += 2) put(xc, e, __fmul2_rn(pair(xc, e), dup(sl2)));
                    } else if (w_left || w_right) {
                        const float2 cv = dup(w_left ? c_left : c_right);
#pragma unroll
                        for (int e = 0; e < KB; e += 2) put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), cv));
                    } else {
                        const int rb = e0 - gi + k;  // table row of element 0, before clamping
#pragma unroll
                        for (int e = 0; e < KB; e += 2) {
                            const float2 rv = make_float2(Rt[min(W - 1, max(0, rb + e)) * BM],
                                                          Rt[min(W - 1, max(0, rb + e + 1)) * BM]);
                            put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), rv));
                        }
                    }
                    if (!full) {  // keys j < nk (and j <= i when causal)
                        const int lim = (CAUSAL ? min(nk, gi + 1) : nk) - e0;
#pragma unroll
                        for (int e = 0; e < KB; ++e) xc[e] = e < lim ? xc[e] : -INFINITY;
                    }
                    rmax = fmaxf(rmax, tc::max32(xc));
                    ptx::tmem_st32f(lb + Tm::S + (uint32_t)(c * KB), xc);
                }
                ptx::tmem_st_wait();  // the stores read x, which the next half overwrites
            }
            // ---- online softmax with a lazy rescale (only when the maximum grows by > 2^8)
            float alpha = 1.f;
            if (rmax > m_ref + kRescaleLog2) {
                alpha = ptx::ex2(m_ref - rmax);  // 0 while nothing was seen yet
                m_ref = rmax;
            }
            // P and O hold the previous tile's product until its P V is done
            if (j >= 1 && !(ok = wait_w(X_PV_DONE, (pv_it + (uint32_t)j - 1u) & 1u))) break;
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                l *= alpha;
                lsum *= alpha;
                if (AV && alpha != 1.f)
                    for (int r = 0; r < W; ++r) Bt[r * BM] *= alpha;
                __syncwarp();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float o[32];
                    ptx::tmem_ld32f(lb + Tm::O + (uint32_t)c0, o);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; e += 2) put(o, e, __fmul2_rn(pair(o, e), dup(alpha)));
                    ptx::tmem_st32f(lb + Tm::O + (uint32_t)c0, o);
                    ptx::tmem_st_wait();
                }
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            // ---- pass 2: exponentials, row sum, value bins, P (bf16 pairs) into TMEM
#pragma unroll 1
            for (int hf = 0; hf < NCH / 2; ++hf) {
                if (2 * hf * KB >= cols) break;  // never read by P V
                float x[2 * KB];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
                    if (2 * hf + cc < live) ptx::tmem_ld32f(lb + Tm::S + (uint32_t)((2 * hf + cc) * KB), x + cc * KB);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * hf + cc;
                    if (c * KB >= cols) continue;
                    float *xc = x + cc * KB;
                    if (c >= live) {  // no row of this warp sees these keys
#pragma unroll
                        for (int e = 0; e < KB / 2; ++e) xc[e] = 0.f;
                    } else {
                        float cst;
                        const bool rawc = raw_chunk(c, cst);
                        const float2 a2 = dup(rawc ? sl2 : 1.f), b2 = dup((rawc ? cst : 0.f) - m_use);
                        float2 s01 = dup(0.f), s23 = dup(0.f);
#pragma unroll
                        for (int e = 0; e < KB; e += 4) {
                            const float2 t0 = __ffma2_rn(pair(xc, e), a2, b2);
                            const float2 t1 = __ffma2_rn(pair(xc, e + 2), a2, b2);
                            xc[e] = ptx::ex2(t0.x);
                            xc[e + 1] = ptx::ex2(t0.y);
                            xc[e + 2] = ptx::ex2(t1.x);
                            xc[e + 3] = ptx::ex2(t1.y);
                            s01 = __fadd2_rn(s01, pair(xc, e));
                            s23 = __fadd2_rn(s23, pair(xc, e + 2));
                        }
                        const float rs = (s01.x + s01.y) + (s23.x + s23.y);
                        l += rs;
                        if (AV) {
                            // bins 1 .. W-2 (causal: 1 .. W-1) receive exactly one key each over
                            // the row and are stored as they come; the end bins come from sums at
                            // the end: bin 0 from l (causal) or from lsum, the keys at or left of
                            // the diagonal
                            const int e0 = j0 + c * KB;
                            if (!CAUSAL) {
                                if (e0 + KB <= gmin) {  // left of every row's diagonal
                                    lsum += rs;
                                } else if (e0 == gmin) {  // the warp's diagonal chunk: keys j <= i
#pragma unroll
                                    for (int e = 0; e < KB; ++e) lsum += e <= lane ? xc[e] : 0.f;
                                }
                            }
                            const bool w_left = (e0 + KB - 1 - gmin) <= -k;
                            const bool w_right = CAUSAL ? e0 > gmax : (e0 - gmax) >= k;
                            if (!w_left && !w_right) {
                                const int rb = e0 - gi + k;  // bin of element 0
#pragma unroll
                                for (int e = 0; e < KB; ++e)
                                    if ((unsigned)(rb + e) < (unsigned)W) Bt[(rb + e) * BM] = xc[e];
                            }
                        }
#pragma unroll
                        for (int e = 0; e < KB / 2; ++e)
                            xc[e] = __uint_as_float(ptx::pack_bf16x2(xc[2 * e], xc[2 * e + 1]));
                    }
                    __syncwarp();
                    ptx::tmem_st16f(lb + Tm::P + (uint32_t)(c * (KB / 2)), xc);
                }
                ptx::tmem_st_wait();  // the stores read x, which the next half overwrites
            }
            // the scores are consumed (S_{j+1} may overwrite them) and P_j is in place
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_S_EMPTY));
            ptx::mbar_arrive(bar(X_P_FULL));
        }
        if (!ok) break;
        pv_it += (uint32_t)J;
        if (AV) {
            // the end bins, then the bins (bf16 pairs) into the S columns: the A operand of
            // O += beta W^V, which the MMA warp issues after the last P V
            if (!CAUSAL && W > 1) {
                // lsum = bin 0 + bins 1 .. k; l - lsum = bins k+1 .. W-2 + bin W-1
                float a = 0.f, b = 0.f;
                for (int r = 1; r <= k; ++r) a += Bt[r * BM];
                for (int r = k + 1; r < W - 1; ++r) b += Bt[r * BM];
                Bt[0] = fmaxf(0.f, lsum - a);
                Bt[(W - 1) * BM] = fmaxf(0.f, (l - lsum) - b);
            } else {  // l = bin 0 + bins 1 .. W-1
                float a = 0.f;
                for (int r = 1; r < W; ++r) a += Bt[r * BM];
                Bt[0] = fmaxf(0.f, l - a);
            }
            for (int c0 = 0; c0 < p.kpad_v; c0 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r0 = c0 + 2 * e;
                    pk[e] = ptx::pack_bf16x2(r0 < W ? Bt[r0 * BM] : 0.f, r0 + 1 < W ? Bt[(r0 + 1) * BM] : 0.f);
                }
                __syncwarp();
                ptx::tmem_st16(lb + Tm::S + (uint32_t)(c0 / 2), pk);
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_BN_FULL));
        }
        // ---- epilogue: O / l -> bf16 into the staging tile (the 128-byte swizzle the output
        // map expects), then one bulk tensor store of the tile (rows past n are not written)
        if (!(ok = wait_w(X_O_FULL, o_it & 1u))) break;
        ++o_it;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        // the O row in halves of 32 columns (four 16-byte chunks each)
        const uint32_t srow = sh.base + p.off_stage + (uint32_t)row * 128u;
#pragma unroll 1
        for (int hc = 0; hc < 2; ++hc) {
            uint32_t r[32];
            ptx::tmem_ld32(lb + Tm::O + (uint32_t)(hc * 32), r);
            ptx::tmem_ld_wait();
            if (hc == 1) {
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(X_O_EMPTY));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 o = __fmul2_rn(make_float2(__uint_as_float(r[8 * q + 2 * h]),
                                                            __uint_as_float(r[8 * q + 2 * h + 1])),
                                                dup(inv));
                    w[h] = ptx::pack_bf16x2(o.x, o.y);
                }
                const int chunk = 4 * hc + q;  // 16-byte chunk of the row, swizzled by row % 8
                ptx::st_shared_v4(srow + (uint32_t)((chunk ^ (row & 7)) * 16), w[0], w[1], w[2], w[3]);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(kSoftBar, 128);
        if (stid == 0) {
            ptx::tma_store_3d(tm_o, sh.base + p.off_stage, 0, qt * BM, bh);
            ptx::bulk_commit();
        }
    }
    // the last tile store has read shared memory and written global memory before the CTA exits
    if (stid == 0) ptx::bulk_wait0();
}

// ======================================================================= kernel
template <bool AK, bool AV, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 2)
    relattn_short_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kf,
                         const __grid_constant__ CUtensorMap tm_vf, const __grid_constant__ CUtensorMap tm_ak,
                         const __grid_constant__ CUtensorMap tm_av, const __grid_constant__ CUtensorMap tm_o,
                         const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    Shared sh;
    sh.base = (raw + 1023u) & ~1023u;
    sh.ptr = smem_raw + (sh.base - raw);
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(sh.ptr + p.off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_ptr + kNumBars);
    sh.abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    sh.limit = p.wait_limit;
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool softmax_arrives = i == X_S_EMPTY || i == X_P_FULL || i == X_BN_FULL || i == X_O_EMPTY;
            ptx::mbar_init(bar_addr(sh, p, i), softmax_arrives ? 128u : 1u);
        }
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_kf);
        ptx::tma_prefetch_desc(&tm_vf);
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_raw = *tmem_slot;

    // each role starts with a full-warp broadcast of the TMEM base, so tcgen05 and TMA
    // operands stay warp-uniform
    if (warp < kSoftWarp0) {
        ptx::reg_dealloc<kCtrlRegs>();
        if (warp == 0) {
            (void)__shfl_sync(0xffffffffu, tmem_raw, 0);
            producer<AK, AV, CAUSAL>(p, sh, &tm_q, &tm_k, &tm_v, &tm_kf, &tm_vf, &tm_ak, &tm_av);
        } else if (warp == 1) {
            mma<AK, AV, CAUSAL>(p, sh, __shfl_sync(0xffffffffu, tmem_raw, 0));
        }
    } else {
        ptx::reg_alloc<kSoftRegs>();
        softmax<AK, AV, CAUSAL>(p, sh, __shfl_sync(0xffffffffu, tmem_raw, 0), &tm_o);
    }
    __syncwarp();

    ptx::tc_fence_before();
    ptx::cta_barrier();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_raw, kTmemCols);
    }
}

}  // namespace sk
}  // namespace relattn
