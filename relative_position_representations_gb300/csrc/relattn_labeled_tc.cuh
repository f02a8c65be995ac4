// Relation-aware attention over labelled edges on the tensor cores, bf16 in / fp32 accumulate,
// for sm_103a ("Self-Attention with Relative Position Representations", section "Relation-Aware
// Self-Attention: The Core Modification": every edge (i, j) carries its own a^K_ij, a^V_ij;
// here the edge's label L_ij picks the table row). In the split form of the paper's section
// 3.4 "Efficient Implementation", with the label in place of clip(j - i, k) + k:
//   e_ij = scale * (q_i . k_j + R_i[L_ij]),      R = Q W^K^T  ([BM x num_labels] per tile),
//   z_i  = sum_j a_ij v_j + sum_l beta_il w^V_l,  beta_il = sum_{j: L_ij = l} a_ij,
// so neither the n x n x d edge tensors nor a per-edge dot product with the tables exists.
//
// One persistent CTA per SM; a work item is one query tile of 128 rows of one head. TMEM holds
// O (D columns at 384) and a ring of three 128-column buffers. Each item makes a sequence of
// buffer "uses": R (with the key table), one score tile S_j = Q K_j^T per key tile, then the
// value bins beta (with the value table). Every use goes through three steps, each ending in
// one arrival on a per-buffer barrier:
//   produce  (MMA warp 1)  R or S_j into the buffer (for beta: nothing)      -> FULL[b]
//   process  (softmax)     R into shared memory / P_j (bf16) over the group's
//                          half of S_j / beta written by group 0             -> P_FULL[b]
//   consume  (MMA warp 2)  nothing / O (+)= P_j V_j / O += beta W^V          -> FREE[b]
// and use u waits for FREE of use u - 3 (the same buffer).
// Warp roles (384 threads), each walking the uses in order:
//   warp 0      TMA loads, K side: Q into one of two buffers, W^K (R), K_j into the K ring.
//   warp 3      TMA loads, V side: V_j into the V ring, W^V (beta W^V).
//   warps 1, 2  MMA issuers of the produce and of the consume steps (one elected lane).
//   warps 4-7   softmax group 0: keys 0..63 of every score tile, output columns 0..D/2-1;
//   warps 8-11  softmax group 1: keys 64..127, output columns D/2..D-1. One thread per query
//               row in each group (TMEM lane = row); the groups keep one running maximum per
//               row (exchanged through shared memory at a named barrier on every tile), so
//               their halves of P enter one P V product; each keeps its own row sum and bins.
//               A thread reads its row's labels of the tile (64 bytes) straight from global
//               memory, issued before it waits for the scores.
// Every wait is bounded; a wait that runs out sets the device status word and the CTA drains
// and exits. The 256 softmax threads take every decision that guards a barrier together.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "relattn_tc_kernel.cuh"

namespace relattn {
namespace lbl {

using tc::BM;
using tc::BN;
using tc::KB;
using tc::kThreads;
using tc::kSoftWarp0;
using tc::kLog2e;
using tc::kRescaleLog2;
using tc::Shared;

constexpr int kSoftThreads = 256;  // both softmax groups
constexpr int kHalf = BN / 2;      // keys of a score tile per group
constexpr int kJointBar = 1;       // hardware named barrier of the 256 softmax threads
constexpr int kNB = 3;             // TMEM buffers in the ring
constexpr int kMaxStages = 4;      // per K or V ring
constexpr int kMaxLabels = 128;    // table rows the tensor-core path stages

struct Params {
    int BH, H, n, n_qtiles, num_items;
    float scale_log2;         // scale * log2(e)
    const int *kv_len;        // [B] or null
    int *err;                 // device status word
    void *out;                // [B, H, n, D] bf16
    const uint8_t *labels;    // [B|1, n, n]
    long long lbs;            // elements between sequences' label matrices (0 = shared)
    int L;                    // table rows (labels)
    int SR, SB;               // shared-memory row strides (floats) of R and of the bins
    int npad_k, kpad_v;       // L rounded up to 16: N of R = Q W^K^T, K of beta W^V
    int table_heads;          // 1: tables indexed by head, 0: one shared table
    uint32_t off_q[2], off_k, off_v, off_ak, off_av, off_r, off_beta[2], off_x, off_bar;
    int kstages, vstages;
    uint32_t kmul, vmul;      // ceil(2^32 / stages) (stages > 1)
    uint32_t stage_bytes;
    long long wait_limit;     // bound of every wait, SM clock cycles
    int lab_vec;              // label rows and matrices start on 16-byte boundaries
};

// TMEM columns (512 allocated): buffer b at 128 b (R: npad_k columns; S_j: 128; a group's P,
// bf16 pairs, over the first 32 of its own 64 score columns; beta: kpad_v / 2), O at 384.
struct Tm {
    static __host__ __device__ constexpr uint32_t buf(uint32_t b) { return 128u * b; }
    static __host__ __device__ constexpr uint32_t P(uint32_t b, uint32_t g) { return 128u * b + 64u * g; }
    static constexpr uint32_t O = 384u;
};

// barriers
enum : int {
    X_Q_FULL = 0,    // two: per Q buffer
    X_Q_EMPTY = 2,   // two
    X_AK_FULL = 4, X_AK_EMPTY, X_AV_FULL, X_AV_EMPTY,
    X_FULL = 8,      // kNB: the buffer's use is produced
    X_PFULL = 11,    // kNB: the softmax has processed it (256 arrivals)
    X_FREE = 14,     // kNB: its consumer MMA is done (the buffer may take the next use)
    X_O_FULL = 17, X_O_EMPTY, X_DRAIN,
    X_KV0 = 20,      // K ring full[kMaxStages], empty[kMaxStages]; V ring the same
    kNumBars = X_KV0 + 4 * kMaxStages
};

__device__ __forceinline__ uint32_t bar_addr(const Shared &sh, const Params &p, int i) {
    return sh.base + p.off_bar + 8u * (uint32_t)i;
}

// position in the ring of TMEM buffers: buffer b, round r (use number = 3 r + b)
struct Slot3 {
    uint32_t b = 0, r = 0;
    __device__ __forceinline__ void next() {
        if (++b == (uint32_t)kNB) {
            b = 0;
            ++r;
        }
    }
};

// allowed keys of the sequence of head bh (before the causal clip)
__device__ __forceinline__ int keys_of(const Params &p, int bh) {
    if (!p.kv_len) return p.n;
    return max(0, min(p.kv_len[bh / p.H], p.n));
}
// keys any row of the tile may see, rounded up to whole 32-key chunks per tile
__device__ __forceinline__ int tile_cols(int nkc, int j) {
    const int c = nkc - j * BN;
    return c >= BN ? BN : ((c + KB - 1) / KB) * KB;
}

// the query tile of item t (longest causal tiles first): head, tile, allowed keys; J = 0 if none
template <bool CAUSAL>
struct Tile {
    int bh, qt, nkc, J;
    __device__ __forceinline__ void make(const Params &p, int t) {
        qt = p.n_qtiles - 1 - t / p.BH;
        bh = t - (p.n_qtiles - 1 - qt) * p.BH;
        const int nk = keys_of(p, bh);
        nkc = CAUSAL ? min(nk, qt * BM + BM) : nk;
        J = (nkc + BN - 1) / BN;
    }
};

// A walk over the uses of the CTA's items (CTA x takes items x, x + gridDim.x, ...; items
// without keys are skipped): use k of an item is R (k = 0, with the key table), S_j, or beta
// (the last, with the value table).
template <bool AK, bool AV, bool CAUSAL>
struct Cursor {
    int i;           // items taken so far
    int t;           // item, or -1 when the walk is over
    Tile<CAUSAL> tl;
    int k, nuse;     // use within the item, uses of the item
    Slot3 s;         // TMEM buffer of the use
    __device__ __forceinline__ explicit Cursor(const Params &p) : i(0) { next_item(p); }
    __device__ __forceinline__ void next_item(const Params &p) {
        k = 0;
        for (;;) {
            t = (int)blockIdx.x + i * (int)gridDim.x;
            ++i;
            if (t >= p.num_items) {
                t = -1;
                break;
            }
            tl.make(p, t);
            if (tl.J > 0) break;
        }
        nuse = (AK ? 1 : 0) + tl.J + (AV ? 1 : 0);
    }
    __device__ __forceinline__ bool valid() const { return t >= 0; }
    __device__ __forceinline__ bool is_r() const { return AK && k == 0; }
    __device__ __forceinline__ bool is_beta() const { return AV && k == nuse - 1; }
    __device__ __forceinline__ int tile() const { return k - (AK ? 1 : 0); }  // S uses
    __device__ __forceinline__ bool first() const { return k == 0; }
    __device__ __forceinline__ bool last() const { return k == nuse - 1; }
    __device__ __forceinline__ void advance(const Params &p) {
        s.next();
        if (++k == nuse) next_item(p);
    }
};

// ring of shared-memory stages
struct Ring {
    uint32_t base;      // shared-memory offset of stage 0
    int stages;
    uint32_t mul;       // ceil(2^32 / stages): e / stages = umulhi(e, mul) (stages > 1)
    int full0, empty0;  // barrier indices of stage 0
};
__device__ __forceinline__ void ring_at(const Ring &r, uint32_t e, uint32_t &st, uint32_t &round) {
    if (r.stages == 1) {  // 2^32 / 1 does not fit the reciprocal
        st = 0;
        round = e;
        return;
    }
    round = __umulhi(e, r.mul);
    st = e - round * (uint32_t)r.stages;
}
__device__ __forceinline__ Ring k_ring(const Params &p) {
    return Ring{p.off_k, p.kstages, p.kmul, X_KV0, X_KV0 + kMaxStages};
}
__device__ __forceinline__ Ring v_ring(const Params &p) {
    return Ring{p.off_v, p.vstages, p.vmul, X_KV0 + 2 * kMaxStages, X_KV0 + 3 * kMaxStages};
}

// ======================================================================= loads
// Two loader warps, each walking the uses in order: warp 0 loads Q (at an item's first use),
// W^K (R) and K_j (S_j) into the K ring; warp 3 loads V_j (P_j V_j) into the V ring and W^V
// (beta W^V). The whole warp runs the role; one elected lane issues.
template <int D, bool AK, bool AV, bool CAUSAL, bool KSIDE>
__device__ void loader(const Params &p, const Shared &sh, const CUtensorMap *tm_q,
                       const CUtensorMap *tm_part, const CUtensorMap *tm_full,
                       const CUtensorMap *tm_tab) {
    constexpr int DB = D / 64;
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    const Ring rg = KSIDE ? k_ring(p) : v_ring(p);
    uint32_t e_it = 0, q_it = 0, t_it = 0;  // ring entries, Q tiles, table loads
    bool ok = true;
    // one K (V) tile of the item into the next stage of the ring
    auto load = [&](const Tile<CAUSAL> &tl, int j) -> bool {
        uint32_t st, round;
        ring_at(rg, e_it, st, round);
        if (!wait(bar(rg.empty0 + (int)st), (round & 1u) ^ 1u)) return false;
        const int nbox = tile_cols(tl.nkc, j) / KB;
        const uint32_t fb = bar(rg.full0 + (int)st);
        ptx::mbar_expect_tx_w(fb, (uint32_t)nbox * KB * D * 2);
        const uint32_t dst = sh.base + rg.base + st * p.stage_bytes;
        if (nbox == BN / KB) {  // whole tile: one box of 128 rows per 64-column block
#pragma unroll
            for (int blk = 0; blk < DB; ++blk)
                ptx::tma_load_3d_w(dst + blk * BN * 128, tm_full, fb, blk * 64, j * BN, tl.bh);
        } else {  // last tile: only the 32-row boxes holding allowed keys
            for (int b = 0; b < nbox; ++b) {
#pragma unroll
                for (int blk = 0; blk < DB; ++blk)
                    ptx::tma_load_3d_w(dst + blk * BN * 128 + b * KB * 128, tm_part, fb, blk * 64,
                                       j * BN + b * KB, tl.bh);
            }
        }
        ++e_it;
        return true;
    };
    Cursor<AK, AV, CAUSAL> cu(p);
    while (ok && cu.valid()) {
        const Tile<CAUSAL> &tl = cu.tl;
        const int th = p.table_heads ? tl.bh % p.H : 0;
        if (KSIDE && cu.first()) {
            const uint32_t qb = q_it & 1u;
            if (!(ok = wait(bar(X_Q_EMPTY + (int)qb), ((q_it >> 1) & 1u) ^ 1u))) break;
            ++q_it;
            ptx::mbar_expect_tx_w(bar(X_Q_FULL + (int)qb), (uint32_t)BM * D * 2);
#pragma unroll
            for (int blk = 0; blk < DB; ++blk)
                ptx::tma_load_3d_w(sh.base + p.off_q[qb] + blk * BM * 128, tm_q, bar(X_Q_FULL + (int)qb),
                                   blk * 64, tl.qt * BM, tl.bh);
        }
        const bool tab = KSIDE ? cu.is_r() : cu.is_beta();
        if (tab) {  // W^K or W^V
            const int fullb = KSIDE ? X_AK_FULL : X_AV_FULL, emptyb = KSIDE ? X_AK_EMPTY : X_AV_EMPTY;
            const int rows = KSIDE ? p.npad_k : p.kpad_v;
            if (!(ok = wait(bar(emptyb), (t_it & 1u) ^ 1u))) break;
            ++t_it;
            ptx::mbar_expect_tx_w(bar(fullb), (uint32_t)rows * D * 2);
            const uint32_t dst = sh.base + (KSIDE ? p.off_ak : p.off_av);
#pragma unroll
            for (int blk = 0; blk < DB; ++blk)
                ptx::tma_load_3d_w(dst + blk * rows * 128, tm_tab, bar(fullb), blk * 64, 0, th);
        } else if (!cu.is_r() && !cu.is_beta()) {
            if (!(ok = load(tl, cu.tile()))) break;
        }
        cu.advance(p);
    }
    // drain: wait (bounded) for the copies issued into shared memory, so that none is still
    // in flight when the CTA exits (normally all were consumed; after an abort the consumers
    // may have given up on some)
    for (uint32_t i = e_it > (uint32_t)rg.stages ? e_it - rg.stages : 0; i < e_it; ++i) {
        uint32_t st, round;
        ring_at(rg, i, st, round);
        tc::drain_bar(bar(rg.full0 + (int)st), round & 1u, sh.limit);
    }
    if (KSIDE)
        for (uint32_t i = q_it > 2u ? q_it - 2u : 0u; i < q_it; ++i)
            tc::drain_bar(bar(X_Q_FULL + (int)(i & 1u)), (i >> 1) & 1u, sh.limit);
    if (t_it) tc::drain_bar(bar(KSIDE ? X_AK_FULL : X_AV_FULL), (t_it - 1) & 1u, sh.limit);
}

// ======================================================================= MMA issuers
// Two MMA warps (the whole warp runs each role with warp-uniform control flow; one elected
// lane issues every tcgen05 instruction), each walking the uses in order: warp 1 produces
// (R, S_j; for beta it only hands the buffer over), warp 2 consumes (P_j V_j, beta W^V; for R
// it only frees the buffer). They meet only through the per-buffer barriers, so neither
// waits while the other's MMAs occupy the tensor pipe.
template <int D, bool AK, bool AV, bool CAUSAL>
__device__ void mma_produce(const Params &p, const Shared &sh, uint32_t tmem) {
    using T = Tm;
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    const Ring rg = k_ring(p);
    const uint64_t dk0 = ptx::sdesc_sw128(sh.base + rg.base, 16, 1024);
    const uint64_t stage16 = p.stage_bytes >> 4;
    // K-major operand, k-step kk of 16: 64-column block kk / 4 (rows x 128 bytes apart),
    // 32 bytes per step inside the 128-byte swizzle atom
    auto kstep = [](int kk, int rows) -> uint64_t {
        return (uint64_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
    };
    uint32_t e_it = 0, q_it = 0, ak_it = 0, qb = 0;
    uint64_t dq = 0;
    bool ok = true;
    Cursor<AK, AV, CAUSAL> cu(p);
    while (ok && cu.valid()) {
        const Tile<CAUSAL> &tl = cu.tl;
        const uint32_t b = cu.s.b;
        if (cu.first()) {
            qb = q_it & 1u;
            if (!(ok = wait(bar(X_Q_FULL + (int)qb), (q_it >> 1) & 1u))) break;
            ++q_it;
            dq = ptx::sdesc_sw128(sh.base + p.off_q[qb], 16, 1024);
        }
        // the buffer's previous use (three uses back) is consumed
        if (cu.s.r > 0 && !(ok = wait(bar(X_FREE + (int)b), (cu.s.r - 1u) & 1u))) break;
        if (cu.is_r()) {  // R = Q W^K^T
            if (!(ok = wait(bar(X_AK_FULL), ak_it & 1u))) break;
            ++ak_it;
            ptx::tc_fence_after();
            const uint32_t idR = ptx::idesc_bf16(BM, (uint32_t)p.npad_k, 0);
            const uint64_t dak = ptx::sdesc_sw128(sh.base + p.off_ak, 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::tc_mma_w(tmem + T::buf(b), dq + kstep(kk, BM), dak + kstep(kk, p.npad_k), idR,
                              kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(bar(X_FULL + (int)b));
            ptx::tc_commit_w(bar(X_AK_EMPTY));  // W^K is free once R is computed
        } else if (cu.is_beta()) {  // nothing to compute: the softmax may write beta
            ptx::tc_fence_after();
            ptx::mbar_arrive_w(bar(X_FULL + (int)b));
        } else {  // S_j = Q K_j^T
            const int j = cu.tile();
            uint32_t stg, round;
            ring_at(rg, e_it, stg, round);
            ++e_it;
            if (!(ok = wait(bar(rg.full0 + (int)stg), round & 1u))) break;
            ptx::tc_fence_after();
            const uint32_t idS = ptx::idesc_bf16(BM, (uint32_t)tile_cols(tl.nkc, j), 0);
            const uint64_t dk = dk0 + (uint64_t)stg * stage16;
            if (D == 128) {
                ptx::tc_mma_ss_k128(tmem + T::buf(b), dq, dk, idS, 0u);
            } else {
                ptx::tc_mma_ss_k64(tmem + T::buf(b), dq, dk, idS, 0u);
            }
            ptx::tc_commit_w(bar(X_FULL + (int)b));
            ptx::tc_commit_w(bar(rg.empty0 + (int)stg));  // K_j is free after it
            if (j == tl.J - 1) ptx::tc_commit_w(bar(X_Q_EMPTY + (int)qb));  // last read of Q
        }
        cu.advance(p);
    }
    // every MMA issued by this warp completes before TMEM is released
    ptx::tc_commit_w(bar(X_DRAIN));
    tc::drain_bar(bar(X_DRAIN), 0, sh.limit);
}

template <int D, bool AK, bool AV, bool CAUSAL>
__device__ void mma_consume(const Params &p, const Shared &sh, uint32_t tmem) {
    using T = Tm;
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = tc::wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    constexpr uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
    const Ring rg = v_ring(p);
    const uint64_t dv0 = ptx::sdesc_sw128(sh.base + rg.base, BN * 128, 1024);
    const uint64_t stage16 = p.stage_bytes >> 4;
    const uint32_t tO = tmem + T::O;
    uint32_t e_it = 0, av_it = 0, o_it = 0;
    bool ok = true;
    Cursor<AK, AV, CAUSAL> cu(p);
    while (ok && cu.valid()) {
        const uint32_t b = cu.s.b;
        if (cu.is_r()) {  // the softmax has copied R out: the buffer is free
            if (!(ok = wait(bar(X_PFULL + (int)b), cu.s.r & 1u))) break;
            ptx::mbar_arrive_w(bar(X_FREE + (int)b));
        } else if (cu.is_beta()) {  // O += beta W^V, beta (bf16 pairs) in the buffer
            if (!(ok = wait(bar(X_AV_FULL), av_it & 1u))) break;
            ++av_it;
            if (!(ok = wait(bar(X_PFULL + (int)b), cu.s.r & 1u))) break;
            ptx::tc_fence_after();
            const uint64_t dav = ptx::sdesc_sw128(sh.base + p.off_av, (uint32_t)p.kpad_v * 128, 1024);
#pragma unroll 1
            for (int kk = 0; kk < p.kpad_v / 16; ++kk)
                ptx::tc_mma_ts_w(tO, tmem + T::buf(b) + (uint32_t)(kk * 8),
                                 dav + (uint64_t)(kk * 16 * 128 >> 4), idPV, 1u);
            ptx::tc_commit_w(bar(X_FREE + (int)b));
            ptx::tc_commit_w(bar(X_AV_EMPTY));
            ptx::tc_commit_w(bar(X_O_FULL));
            ++o_it;
        } else {  // O (+)= P_j V_j, P over the buffer
            const int j = cu.tile();
            uint32_t stg, round;
            ring_at(rg, e_it, stg, round);
            ++e_it;
            if (!(ok = wait(bar(rg.full0 + (int)stg), round & 1u))) break;
            // the first product of an item overwrites O: the previous item's O is read out
            if (j == 0 && !(ok = wait(bar(X_O_EMPTY), (o_it & 1u) ^ 1u))) break;
            if (!(ok = wait(bar(X_PFULL + (int)b), cu.s.r & 1u))) break;
            ptx::tc_fence_after();
            const int cols = tile_cols(cu.tl.nkc, j);
            const uint64_t dv = dv0 + (uint64_t)stg * stage16;
            const uint32_t a_lo = tmem + T::P(b, 0), a_hi = tmem + T::P(b, 1);
            const int nk16 = cols / 16;
            if (nk16 == BN / 16) {  // a whole tile: one chain of 8 k-steps
                ptx::tc_mma_ts_k128_2(tO, a_lo, a_hi, dv, idPV, j > 0 ? 1u : 0u);
            } else {
#pragma unroll 1
                for (int kk = 0; kk < nk16; ++kk)
                    ptx::tc_mma_ts_w(tO, (kk < 4 ? a_lo : a_hi) + (uint32_t)((kk & 3) * 8),
                                     dv + (uint64_t)(kk * 16 * 128 >> 4), idPV,
                                     (j > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::tc_commit_w(bar(X_FREE + (int)b));
            ptx::tc_commit_w(bar(rg.empty0 + (int)stg));  // V_j is free after it
            if (cu.last()) {
                ptx::tc_commit_w(bar(X_O_FULL));
                ++o_it;
            }
        }
        cu.advance(p);
    }
    // every MMA issued by this warp completes before TMEM is released
    ptx::tc_commit_w(bar(X_DRAIN));
    tc::drain_bar(bar(X_DRAIN), 0, sh.limit);
}


// ======================================================================= softmax / epilogue
// Group g (warps 4 + 4g .. 7 + 4g) of the 256 softmax threads: score chunks 2g and 2g + 1 (32
// keys each) of every tile, output columns g D/2 .. g D/2 + D/2 - 1; thread = query row.
template <int D, bool AK, bool AV, bool CAUSAL>
__device__ void softmax(const Params &p, const Shared &sh, uint32_t tmem, int grp_in) {
    using T = Tm;
    using tc::pair;
    using tc::put;
    using tc::dup;
    const int g = __shfl_sync(0xffffffffu, grp_in, 0);  // known warp-uniform from here on
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto uni = [](int v) { return __shfl_sync(0xffffffffu, v, 0); };
    const int quad = uni(warp & 3);  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    auto bar = [&](int i) { return bar_addr(sh, p, i); };
    float *Rrow = reinterpret_cast<float *>(sh.ptr + p.off_r) + row * p.SR;
    float *brow = reinterpret_cast<float *>(sh.ptr + p.off_beta[g]) + row * p.SB;
    const float *brow1 = reinterpret_cast<const float *>(sh.ptr + p.off_beta[1]) + row * p.SB;
    float *mx = reinterpret_cast<float *>(sh.ptr + p.off_x);                  // [2][2][128]
    float2 *xl = reinterpret_cast<float2 *>(sh.ptr + p.off_x + 2 * 2 * BM * 4);  // [2][128]
    const float sl2 = p.scale_log2;
    const int W = p.L;
    uint32_t o_it = 0, par = 0;
    Slot3 sl;  // TMEM buffer of the current use
    bool ok = true, bad = false;
    // A wait of all 256 softmax threads: warp 4 polls the mbarrier, the others meet it at the
    // joint named barrier, whose AND-reduction carries the outcome to every thread.
    auto jwait = [&](uint32_t b, uint32_t parity) -> bool {
        bool r = true;
        if (warp == kSoftWarp0) {
            r = tc::wait_bar(b, parity, sh, p.err);
            r = __all_sync(0xffffffffu, r ? 1 : 0) != 0;
        }
        return ptx::bar_red_and(kJointBar, kSoftThreads, r);
    };
    auto jsync = [&]() { ptx::named_bar_sync(kJointBar, kSoftThreads); };

    for (int it = 0;; ++it) {
        const int t = (int)blockIdx.x + it * (int)gridDim.x;
        if (t >= p.num_items || !ok) break;
        Tile<CAUSAL> tl;
        tl.make(p, t);
        const int bh = uni(tl.bh), qt = uni(tl.qt);
        const int i0 = qt * BM, gi = i0 + row;
        const int gmax = uni(i0 + quad * 32) + 31;  // last row of this warp
        const int nk = uni(keys_of(p, bh));
        const int nkc = uni(tl.nkc);  // keys any row of the tile may see
        const int J = uni(tl.J);
        __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                              ((long long)bh * p.n + gi) * D + g * (D / 2);
        if (J == 0) {  // no allowed key: the rows are zero (no MMA, no barrier for this item)
            if (gi < p.n) {
#pragma unroll
                for (int c = 0; c < D / 16; ++c)
                    reinterpret_cast<uint4 *>(orow)[c] = make_uint4(0, 0, 0, 0);
            }
            continue;
        }
        // this row's labels (rows beyond n read the last row; they are never stored; without a
        // table the labels are not read)
        const uint8_t *lrow = (AK || AV) ? p.labels + (long long)(bh / p.H) * p.lbs +
                                               (long long)min(gi, p.n - 1) * p.n
                                         : nullptr;
        if (AK) {  // use R: the row -> shared memory (scaled to the log2 domain), half per group
            if (!(ok = jwait(bar(X_FULL + (int)sl.b), sl.r & 1u))) break;
            ptx::tc_fence_after();
            for (int c0 = 16 * g; c0 < p.npad_k; c0 += 32) {
                uint32_t r[16];
                ptx::tmem_ld16(lane_base + T::buf(sl.b) + (uint32_t)c0, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c0 + e < W) Rrow[c0 + e] = __uint_as_float(r[e]) * sl2;
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_PFULL + (int)sl.b));
            sl.next();
            jsync();  // the whole row is in shared memory
        }
        if (AV)
            for (int r = 0; r < W; ++r) brow[r] = 0.f;
        float m_ref = -INFINITY, l = 0.f;
        const int cbase = 2 * g;  // this group's first chunk of a tile
        Slot3 prev;  // buffer of the previous score tile

        for (int j = 0; j < J; ++j) {
            const uint32_t b = sl.b;
            const int j0 = j * BN;
            const int kg = j0 + cbase * KB;  // first key of this group
            const int cols = tile_cols(nkc, j);  // multiple of 32, > 0
            int live = max(0, min(2, cols / KB - cbase));  // this group's chunks any row sees
            if (CAUSAL) live = min(live, max(0, (gmax - kg) / KB + 1));
            // the labels of this group's 64 keys (issued before the wait for the scores);
            // keys beyond n read as label 0 (they are masked)
            uint32_t lw[kHalf / 4];
            if (!(AK || AV)) {
#pragma unroll
                for (int q = 0; q < kHalf / 4; ++q) lw[q] = 0;
            } else if (p.lab_vec) {
#pragma unroll
                for (int q = 0; q < kHalf / 16; ++q) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (kg + 16 * q < p.n) v = *reinterpret_cast<const uint4 *>(lrow + kg + 16 * q);
                    lw[4 * q] = v.x;
                    lw[4 * q + 1] = v.y;
                    lw[4 * q + 2] = v.z;
                    lw[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < kHalf / 4; ++q) {
                    uint32_t w4 = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (kg + 4 * q + e < p.n) w4 |= (uint32_t)lrow[kg + 4 * q + e] << (8 * e);
                    lw[q] = w4;
                }
            }
            if (!(ok = jwait(bar(X_FULL + (int)b), sl.r & 1u))) break;
            ptx::tc_fence_after();
            // ---- this group's half of the score row: chunk kinds (warp-uniform) beyond the
            // loaded columns (no P), seen by no row of the warp (P = 0), or full logits
            enum { kDead = 0, kNone = 1, kFull = 3 };
            int kind[2];
            float x[kHalf];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = cbase + cc;
                kind[cc] = uni(c * KB >= cols ? kDead : cc >= live ? kNone : kFull);
                if (kind[cc] == kFull)
                    ptx::tmem_ld32f(lane_base + T::buf(b) + (uint32_t)(c * KB), x + cc * KB);
            }
            ptx::tmem_ld_wait();
            // ---- logits in the log2 domain: scale * (q.k + R[label]), masks; labels without a
            // table row read as the last row and are reported
            float rmax = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                float *xc = x + cc * KB;
                if (kind[cc] != kFull) {
#pragma unroll
                    for (int e = 0; e < KB; ++e) xc[e] = -INFINITY;
                    continue;
                }
                const int e0 = kg + cc * KB;
                const int lim = (CAUSAL ? min(nk, gi + 1) : nk) - e0;  // keys e < lim are allowed
#pragma unroll
                for (int e = 0; e < KB; ++e) {
                    if (AK || AV) {
                        const int lb = (int)((lw[(cc * KB + e) >> 2] >> (8 * (e & 3))) & 0xffu);
                        bad |= e < lim && lb >= W;
                    }
                }
                if (AK) {
#pragma unroll
                    for (int e = 0; e < KB; e += 2) {
                        const int l0 = min(W - 1, (int)((lw[(cc * KB + e) >> 2] >> (8 * (e & 3))) & 0xffu));
                        const int l1 = min(W - 1, (int)((lw[(cc * KB + e + 1) >> 2] >> (8 * ((e + 1) & 3))) & 0xffu));
                        put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), make_float2(Rrow[l0], Rrow[l1])));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < KB; e += 2) put(xc, e, __fmul2_rn(pair(xc, e), dup(sl2)));
                }
#pragma unroll
                for (int e = 0; e < KB; ++e) xc[e] = e < lim ? xc[e] : -INFINITY;
                rmax = fmaxf(rmax, tc::max32(xc));
            }
            // ---- one running maximum for both groups: exchange the tile maxima of the row
            // (two buffers by tile parity: a group is never more than one barrier ahead). The
            // OR-reduction tells whether any row of the tile grows its maximum by more than
            // 2^8, i.e. whether O has to be rescaled.
            mx[(par * 2 + (uint32_t)g) * BM + row] = rmax;
            const bool any = ptx::bar_red_or(kJointBar, kSoftThreads, rmax > m_ref + kRescaleLog2);
            rmax = fmaxf(rmax, mx[(par * 2 + (uint32_t)(1 - g)) * BM + row]);
            par ^= 1u;
            // ---- online softmax with a lazy rescale
            float alpha = 1.f;
            if (rmax > m_ref + kRescaleLog2) {
                alpha = ptx::ex2(m_ref - rmax);  // 0 while nothing was seen yet
                m_ref = rmax;
            }
            if (any && j >= 1) {
                // O holds P_{<j} V: it is rescaled only once P_{j-1} V_{j-1} has completed
                if (!(ok = jwait(bar(X_FREE + (int)prev.b), prev.r & 1u))) break;
                ptx::tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    l *= alpha;
                    if (AV && alpha != 1.f)
                        for (int r = 0; r < W; ++r) brow[r] *= alpha;
                    __syncwarp();
#pragma unroll
                    for (int c0 = 0; c0 < D / 2; c0 += 32) {  // this group's half of O
                        uint32_t r[32];
                        const uint32_t ta = lane_base + T::O + (uint32_t)(g * (D / 2) + c0);
                        ptx::tmem_ld32(ta, r);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v = __fmul2_rn(
                                make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), dup(alpha));
                            r[e] = __float_as_uint(v.x);
                            r[e + 1] = __float_as_uint(v.y);
                        }
                        ptx::tmem_st32(ta, r);
                    }
                    ptx::tmem_st_wait();
                }
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            // ---- exponentials (masked and unseen keys hold -inf: 0), row sum
#pragma unroll
            for (int e = 0; e < kHalf; e += 2) {
                const float2 t = __fadd2_rn(pair(x, e), dup(-m_use));
                x[e] = ptx::ex2(t.x);
                x[e + 1] = ptx::ex2(t.y);
            }
            float2 s4[4] = {dup(0.f), dup(0.f), dup(0.f), dup(0.f)};
#pragma unroll
            for (int e = 0; e < kHalf; e += 8) {
                s4[0] = __fadd2_rn(s4[0], pair(x, e));
                s4[1] = __fadd2_rn(s4[1], pair(x, e + 2));
                s4[2] = __fadd2_rn(s4[2], pair(x, e + 4));
                s4[3] = __fadd2_rn(s4[3], pair(x, e + 6));
            }
            {
                const float2 u = __fadd2_rn(__fadd2_rn(s4[0], s4[1]), __fadd2_rn(s4[2], s4[3]));
                l += u.x + u.y;
            }
            // ---- value bins: beta_il += p_ij for the label of every key (this group's own
            // array; a masked key adds 0)
            if (AV) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    if (kind[cc] != kFull) continue;
#pragma unroll
                    for (int e = 0; e < KB; ++e) {
                        const int lb = min(W - 1, (int)((lw[(cc * KB + e) >> 2] >> (8 * (e & 3))) & 0xffu));
                        brow[lb] += x[cc * KB + e];
                    }
                }
            }
            // ---- P (bf16 pairs) into TMEM over this group's own score columns (already read)
#pragma unroll
            for (int e = 0; e < kHalf / 2; ++e) x[e] = __uint_as_float(ptx::pack_bf16x2(x[2 * e], x[2 * e + 1]));
            __syncwarp();
            if (kind[1] != kDead)
                ptx::tmem_st32f(lane_base + T::P(b, (uint32_t)g), x);
            else if (kind[0] != kDead)
                ptx::tmem_st16f(lane_base + T::P(b, (uint32_t)g), x);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_PFULL + (int)b));
            prev = sl;
            sl.next();
        }
        if (!ok) break;
        // ---- the two groups' row sums, added
        xl[g * BM + row] = make_float2(l, 0.f);
        if (AV) {  // use beta: wait for the buffer (its joint barrier also publishes xl)
            if (!(ok = jwait(bar(X_FULL + (int)sl.b), sl.r & 1u))) break;
            ptx::tc_fence_after();
            l += xl[(1 - g) * BM + row].x;
            if (g == 0) {
                // beta = the bins of both groups. Group 1's array is read here and cleared only
                // after the epilogue's joint wait, which comes after this group's arrival below.
                for (int c0 = 0; c0 < p.kpad_v; c0 += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r0 = c0 + 2 * e;
                        const float lo = r0 < W ? brow[r0] + brow1[r0] : 0.f;
                        const float hi = r0 + 1 < W ? brow[r0 + 1] + brow1[r0 + 1] : 0.f;
                        pk[e] = ptx::pack_bf16x2(lo, hi);
                    }
                    __syncwarp();
                    ptx::tmem_st16(lane_base + T::buf(sl.b) + (uint32_t)(c0 / 2), pk);
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(X_PFULL + (int)sl.b));
            sl.next();
        }
        // ---- epilogue: O / l -> bf16 -> global, this group's half of the columns
        if (!(ok = jwait(bar(X_O_FULL), o_it & 1u))) break;
        ++o_it;
        ptx::tc_fence_after();
        if (!AV) l += xl[(1 - g) * BM + row].x;  // written before the joint wait's barrier
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld32(lane_base + T::O + (uint32_t)(g * (D / 2) + c0), r);
            ptx::tmem_ld_wait();
            if (gi < p.n) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w4[4];
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        const float2 o = __fmul2_rn(make_float2(__uint_as_float(r[8 * q + 2 * hh]),
                                                                __uint_as_float(r[8 * q + 2 * hh + 1])),
                                                    dup(inv));
                        w4[hh] = ptx::pack_bf16x2(o.x, o.y);
                    }
                    reinterpret_cast<uint4 *>(orow)[c0 / 8 + q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
            __syncwarp();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(X_O_EMPTY));
    }
    // a label without a table row was read (as the last row): report it
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(p.err, 0, (int)kLabelOutOfRange);
}

// ======================================================================= kernel
template <int D, bool AK, bool AV, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    relattn_labeled_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kf,
                              const __grid_constant__ CUtensorMap tm_vf, const __grid_constant__ CUtensorMap tm_ak,
                              const __grid_constant__ CUtensorMap tm_av, const __grid_constant__ Params p) {
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
            uint32_t cnt = 1;
            if ((i >= X_PFULL && i < X_PFULL + kNB) || i == X_O_EMPTY)
                cnt = kSoftThreads;  // both softmax groups
            if (i == X_DRAIN) cnt = 2;  // both MMA warps
            ptx::mbar_init(bar_addr(sh, p, i), cnt);
        }
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_kf);
        ptx::tma_prefetch_desc(&tm_vf);
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_raw = *tmem_slot;

    // Each role starts with a full-warp broadcast of the TMEM base: it tells the compiler the
    // warp is converged and the value warp-uniform.
    if (warp == 0 || warp == 3) {  // loaders: K side (Q, W^K, K ring), V side (V ring, W^V)
        (void)__shfl_sync(0xffffffffu, tmem_raw, 0);
        if (warp == 0)
            loader<D, AK, AV, CAUSAL, true>(p, sh, &tm_q, &tm_k, &tm_kf, &tm_ak);
        else
            loader<D, AK, AV, CAUSAL, false>(p, sh, &tm_q, &tm_v, &tm_vf, &tm_av);
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_raw, 0);
        if (warp == 1)
            mma_produce<D, AK, AV, CAUSAL>(p, sh, tmem);
        else
            mma_consume<D, AK, AV, CAUSAL>(p, sh, tmem);
        __syncwarp();
    } else {
        const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_raw, 0);
        softmax<D, AK, AV, CAUSAL>(p, sh, tmem, (warp - kSoftWarp0) >> 2);
    }

    ptx::tc_fence_before();
    ptx::cta_barrier();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_raw, 512);
    }
}

}  // namespace lbl
}  // namespace relattn
