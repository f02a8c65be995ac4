// Fused relation-aware attention forward, bf16 in / fp32 accumulate, for sm_103a.
//
// Method: Shaw, Uszkoreit & Vaswani (paper summary page, section 3.4): eq. 4 in the split
// form of eq. 5,
//   e_ij = scale * (q_i . k_j + R_i[clip(j-i,k)+k]),    R = Q W^K^T  ([BM x (2k+1)] per tile),
// and eq. 3 split in two sums,
//   z_i = sum_j a_ij v_j + sum_r beta_ir w^V_r,   beta_ir = sum_{j: clip(j-i,k)+k = r} a_ij.
// T5 variant ("Relative position embeddings", section "T5"): e_ij = scale*q_i.k_j + b[bucket].
//
// Persistent CTAs (one or two per SM) loop over work items (query tile of 128 rows, head),
// longest causal rows first. Warp roles:
//   warp 0      TMA producer: Q tile and edge tables, then K/V tiles of 128 keys (in boxes of
//               32 rows, none past the last allowed key) into a ring of stages, in the order
//               the MMA warp consumes them (K0 K1 V0 K2 V1 ...), and W^V at the end.
//   warp 1      MMA issuer (one thread). Per tile: R = Q W^K^T into a score buffer, then
//               S_j = Q K_j^T into the score buffer(s), O += P_j V_j with P read from TMEM,
//               and at the end O += beta W^V with the bins read from TMEM.
//   warps 2..   softmax / epilogue: each query row (= TMEM lane) is handled by NSPLIT
//               threads (one per 64 keys of a key tile; the two halves of a 128-key tile
//               exchange their row maxima through shared memory). Per key tile: add the
//               relative term (a per-row constant for 32-key chunks that lie beyond +-k for
//               the whole warp, a shared-memory gather inside the band), mask, online softmax
//               in the exp2 domain with a lazy rescale (only when the running max grows by
//               more than 2^8), value bins, bf16 P into TMEM. Chunks no row of the warp can
//               see are skipped. Epilogue: O / l -> bf16.
// Score (S) and probability (P) tiles are double-buffered in TMEM, so S_{j+1} and the
// P_{j-1} V_{j-1} product overlap the softmax of tile j.
// TMEM: CPS = 1 (one CTA per SM, 128-key tiles): S0 [0,128) S1 [128,256) O [256,256+D)
//       P0 [384,448) P1 [448,512);
//       CPS = 2 (two CTAs per SM, D = 64, 64-key tiles): S0 [0,64) S1 [64,128) P0 [128,160)
//       P1 [160,192) O [192,256).
// Every wait is bounded; a wait that runs out sets the device status word and the CTA
// drains and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "relattn_internal.h"
#include "sm103_ptx.cuh"

namespace relattn {
namespace tc {

constexpr int BM = 128;   // query rows per tile (= TMEM lanes)
constexpr int KB = 32;    // key rows per TMA box and keys per softmax chunk
constexpr int HC = 64;    // keys of a key tile handled by one softmax thread
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
// bound of every device wait, in SM clock cycles (about one second at 2 GHz); clock64 is
// read only after a wait did not succeed at once and then every 256 polls
constexpr long long kWaitLimitCycles = 2000000000ll;

template <int CPS>
struct TmemLayout {
    static constexpr int BN = CPS == 1 ? 128 : 64;  // keys per key tile
    static constexpr int NSPLIT = BN / HC;          // softmax threads per query row
    // registers are allocated per 4-warp group: two CTAs per SM need whole warpgroups
    // (warps 2-3 idle) to stay within 128 registers a thread
    static constexpr int SW0 = CPS == 2 ? 4 : 2;     // first softmax warp
    static constexpr int THREADS = 32 * SW0 + 128 * NSPLIT;
    static constexpr uint32_t cols = CPS == 1 ? 512u : 256u;
    static constexpr uint32_t S = 0;                         // S buffer b at S + b * BN
    static constexpr uint32_t O = CPS == 1 ? 256u : 192u;    // D columns
    static constexpr uint32_t P = CPS == 1 ? 384u : 128u;    // P buffer b at P + b * BN / 2
};

// barrier slots
enum : int {
    B_Q_FULL = 0, B_Q_EMPTY, B_S_FULL0, B_S_FULL1, B_S_EMPTY0, B_S_EMPTY1, B_P_FULL0, B_P_FULL1,
    B_PV_DONE0, B_PV_DONE1, B_AV_FULL, B_AV_EMPTY, B_O_FULL, B_DRAIN, B_GROUP, B_PAIR0,
    B_KV0 = B_PAIR0 + 4
};
constexpr int kMaxStages = 8;
constexpr int kNumBars = B_KV0 + 2 * kMaxStages;

struct Params {
    int BH, H, n;
    int n_qtiles, num_tiles;
    float scale_log2;   // scale * log2(e)
    const int *kv_len;  // [B] or null
    int *err;           // device status word
    void *out;          // [B, H, n, D] bf16
    int clip_k;         // Shaw: k
    int W;              // table rows staged: k+1 (causal) or 2k+1
    int SR;             // row stride (floats) of the per-row tables in shared memory
    int npad_k;         // W rounded up to 16: N of the R = Q W^K^T MMA
    int kpad_v;         // W rounded up to 16: K of the beta W^V MMA
    int table_heads;    // 1: tables indexed by head, 0: one shared table
    const float *bias;  // T5 [num_buckets, H]
    int t5_R;           // T5 offset-table radius (bucket is constant beyond it)
    T5Buckets t5;
    uint32_t off_q, off_kv, off_ak, off_av, off_r, off_beta, off_t5, off_x, off_bar;
    int stages;
    uint32_t stage_bytes;
    int head_group;     // heads whose tiles are scheduled together (K/V reuse in L2)
};

struct Shared {
    uint32_t base;  // 1024-aligned shared address
    uint8_t *ptr;   // generic pointer to the same byte
    volatile int *abort_flag;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Shared &sh,
                                         int *err) {
    if (ptx::mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try(bar, parity)) return true;
        if ((++spins & 255u) == 0) {
            if (*sh.abort_flag) return false;
            if (clock64() - t0 > kWaitLimitCycles) {
                *sh.abort_flag = 1;
                atomicCAS(err, 0, 4 /* RELATTN_ERR_TIMEOUT */);
                return false;
            }
        }
    }
}

// bounded poll of a barrier during teardown (no abort check)
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!ptx::mbar_try(bar, parity) && clock64() - t0 < kWaitLimitCycles) {
    }
}

// Barrier among the 128 softmax threads on an mbarrier, so the wait stays bounded (a plain
// bar.sync would hang if a thread of the group left after a timeout). Warp-uniform result.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t &it, const Shared &sh, int *err) {
    ptx::mbar_arrive(bar);
    const bool ok = wait_bar(bar, it & 1u, sh, err);
    ++it;
    return __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
}

// Work order: heads in groups of head_group (their K/V stay in L2 while the group runs);
// inside a group, the query tiles with the most keys (causal) come first.
__device__ __forceinline__ void decode_tile(const Params &p, int t, int &bh, int &qt) {
    const int per_group = p.head_group * p.n_qtiles;
    const int g = t / per_group, r = t - g * per_group;
    const int g0 = g * p.head_group;
    const int gsize = min(p.head_group, p.BH - g0);
    qt = p.n_qtiles - 1 - r / gsize;
    bh = g0 + r % gsize;
}

// number of allowed keys (before the causal clip) of the sequence of head bh
__device__ __forceinline__ int keys_of(const Params &p, int bh) {
    if (!p.kv_len) return p.n;
    return max(0, min(p.kv_len[bh / p.H], p.n));
}

// keys any row of query tile i0 may see
template <bool CAUSAL>
__device__ __forceinline__ int tile_keys(const Params &p, int bh, int i0) {
    const int nk = keys_of(p, bh);
    return CAUSAL ? min(nk, i0 + BM) : nk;
}

// columns of key tile j that are loaded and multiplied: the allowed keys rounded up to
// whole 32-row boxes
template <int BN>
__device__ __forceinline__ int tile_cols(int nkc, int j) {
    const int c = nkc - j * BN;
    return c >= BN ? BN : ((c + KB - 1) / KB) * KB;
}

// ======================================================================= producer
template <int D, bool AK, bool AV, bool CAUSAL, int CPS>
__device__ void producer_role(const Params &p, const Shared &sh, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                              const CUtensorMap *tm_kf, const CUtensorMap *tm_vf,
                              const CUtensorMap *tm_ak, const CUtensorMap *tm_av) {
    constexpr int DB = D / 64;
    constexpr int BN = TmemLayout<CPS>::BN;
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    const uint32_t sQ = sh.base + p.off_q, sKV = sh.base + p.off_kv;
    const uint32_t sAK = sh.base + p.off_ak, sAV = sh.base + p.off_av;
    const int S = p.stages;
    uint32_t kv_it = 0, q_it = 0, av_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int bh, qt;
        decode_tile(p, t, bh, qt);
        const int i0 = qt * BM, h = bh % p.H;
        const int nkc = tile_keys<CAUSAL>(p, bh, i0);
        const int J = (nkc + BN - 1) / BN;
        if (J == 0) continue;
        if (!(ok = wait_bar(bar(B_Q_EMPTY), (q_it & 1u) ^ 1u, sh, p.err))) break;
        const uint32_t qbytes = (uint32_t)BM * D * 2 + (AK ? (uint32_t)p.npad_k * D * 2 : 0u);
        ptx::mbar_expect_tx(bar(B_Q_FULL), qbytes);
#pragma unroll
        for (int blk = 0; blk < DB; ++blk)
            ptx::tma_load_3d(sQ + blk * BM * 128, tm_q, bar(B_Q_FULL), blk * 64, i0, bh);
        if (AK) {
#pragma unroll
            for (int blk = 0; blk < DB; ++blk)
                ptx::tma_load_3d(sAK + blk * p.npad_k * 128, tm_ak, bar(B_Q_FULL), blk * 64, 0,
                                 p.table_heads ? h : 0);
        }
        ++q_it;
        // K/V tiles in consumption order: K0, K1, V0, K2, V1, ..., K_{J-1}, V_{J-2}, V_{J-1}
        for (int s = 0; s < 2 * J; ++s) {
            int j;
            bool isK;
            if (s == 0) { j = 0; isK = true; }
            else if (s == 2 * J - 1) { j = J - 1; isK = false; }
            else if (s & 1) { j = (s + 1) >> 1; isK = true; }
            else { j = (s >> 1) - 1; isK = false; }
            const int st = (int)(kv_it % (uint32_t)S);
            const uint32_t round = kv_it / (uint32_t)S;
            if (!(ok = wait_bar(bar(B_KV0 + kMaxStages + st), (round & 1u) ^ 1u, sh, p.err))) break;
            const int nbox = tile_cols<BN>(nkc, j) / KB;
            ptx::mbar_expect_tx(bar(B_KV0 + st), (uint32_t)nbox * KB * D * 2);
            const uint32_t dst = sKV + (uint32_t)st * p.stage_bytes;
            if (nbox == BN / KB) {  // whole tile: one box of BN rows per 64-column block
#pragma unroll
                for (int blk = 0; blk < DB; ++blk)
                    ptx::tma_load_3d(dst + blk * BN * 128, isK ? tm_kf : tm_vf, bar(B_KV0 + st),
                                     blk * 64, j * BN, bh);
            } else {  // last tile: only the 32-row boxes holding allowed keys
                for (int b = 0; b < nbox; ++b) {
#pragma unroll
                    for (int blk = 0; blk < DB; ++blk)
                        ptx::tma_load_3d(dst + blk * BN * 128 + b * KB * 128, isK ? tm_k : tm_v,
                                         bar(B_KV0 + st), blk * 64, j * BN + b * KB, bh);
                }
            }
            ++kv_it;
        }
        if (!ok) break;
        if (AV) {
            if (!(ok = wait_bar(bar(B_AV_EMPTY), (av_it & 1u) ^ 1u, sh, p.err))) break;
            ptx::mbar_expect_tx(bar(B_AV_FULL), (uint32_t)p.kpad_v * D * 2);
#pragma unroll
            for (int blk = 0; blk < DB; ++blk)
                ptx::tma_load_3d(sAV + blk * p.kpad_v * 128, tm_av, bar(B_AV_FULL), blk * 64, 0,
                                 p.table_heads ? h : 0);
            ++av_it;
        }
    }
    if (!ok) {
        // drain: wait (bounded) for copies already issued into shared memory
        for (uint32_t it = kv_it > (uint32_t)S ? kv_it - S : 0; it < kv_it; ++it)
            drain_bar(bar(B_KV0 + (int)(it % (uint32_t)S)), (it / (uint32_t)S) & 1u);
        if (q_it) drain_bar(bar(B_Q_FULL), (q_it - 1) & 1u);
        if (AV && av_it) drain_bar(bar(B_AV_FULL), (av_it - 1) & 1u);
    }
}

// ======================================================================= MMA issuer
template <int D, bool AK, bool AV, bool CAUSAL, int CPS>
__device__ void mma_role(const Params &p, const Shared &sh, uint32_t tmem) {
    using TL = TmemLayout<CPS>;
    constexpr int BN = TL::BN;
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    const uint32_t sQ = sh.base + p.off_q, sKV = sh.base + p.off_kv;
    const uint32_t sAK = sh.base + p.off_ak, sAV = sh.base + p.off_av;
    const int S = p.stages;
    uint32_t kv_it = 0, q_it = 0, av_it = 0, s_it = 0, p_it = 0;
    bool ok = true;

    // the next score-buffer item (R or S_j): wait until the softmax released the buffer
    auto next_sbuf = [&](uint32_t &col, uint32_t &fullbar) -> bool {
        const uint32_t buf = s_it & 1u;
        const uint32_t use = s_it >> 1;
        if (!wait_bar(bar(B_S_EMPTY0 + (int)buf), (use & 1u) ^ 1u, sh, p.err)) return false;
        ptx::tc_fence_after();
        col = TL::S + buf * BN;
        fullbar = bar(B_S_FULL0 + (int)buf);
        ++s_it;
        return true;
    };

    // O += P_j V_j: P from TMEM buffer (item & 1) as bf16 pairs, V tile MN-major in shared
    // memory. Completion is signalled on the buffer's own barrier.
    // Each P buffer has its own full barrier: the softmax may run one item ahead, and a
    // shared barrier could then complete twice before this thread waits on it.
    auto wait_p = [&](uint32_t &pb) -> bool {
        pb = p_it & 1u;
        if (!wait_bar(bar(B_P_FULL0 + (int)pb), (p_it >> 1) & 1u, sh, p.err)) return false;
        ++p_it;
        return true;
    };
    auto issue_pv = [&](int j, int cols) -> bool {
        uint32_t pb;
        if (!wait_p(pb)) return false;
        const int st = (int)(kv_it % (uint32_t)S);
        if (!wait_bar(bar(B_KV0 + st), (kv_it / (uint32_t)S) & 1u, sh, p.err)) return false;
        ptx::tc_fence_after();
        const uint32_t vb = sKV + (uint32_t)st * p.stage_bytes;
        const uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
        const uint32_t pcol = TL::P + pb * (BN / 2);
        for (int kk = 0; kk < cols / 16; ++kk) {
            const uint64_t b = ptx::sdesc_sw128(vb + kk * 16 * 128, BN * 128, 1024);
            ptx::tc_mma_ts(tmem + TL::O, tmem + pcol + (uint32_t)(kk * 8), b, idPV,
                           (j > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::tc_commit(bar(B_PV_DONE0 + (int)pb));
        ptx::tc_commit(bar(B_KV0 + kMaxStages + st));
        ++kv_it;
        return true;
    };

    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int bh, qt;
        decode_tile(p, t, bh, qt);
        const int nkc = tile_keys<CAUSAL>(p, bh, qt * BM);
        const int J = (nkc + BN - 1) / BN;
        if (J == 0) continue;
        if (!(ok = wait_bar(bar(B_Q_FULL), q_it & 1u, sh, p.err))) break;
        ++q_it;
        ptx::tc_fence_after();
        if (AK) {
            uint32_t col, fb;
            if (!(ok = next_sbuf(col, fb))) break;
            const uint32_t idR = ptx::idesc_bf16(BM, (uint32_t)p.npad_k, 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = ptx::sdesc_sw128(sQ + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
                const uint64_t b =
                    ptx::sdesc_sw128(sAK + (kk >> 2) * p.npad_k * 128 + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma(tmem + col, a, b, idR, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit(fb);
        }
        int prev_cols = 0;
        for (int j = 0; j < J && ok; ++j) {
            const int cols = tile_cols<BN>(nkc, j);
            const int st = (int)(kv_it % (uint32_t)S);
            if (!(ok = wait_bar(bar(B_KV0 + st), (kv_it / (uint32_t)S) & 1u, sh, p.err))) break;
            uint32_t col, fb;
            if (!(ok = next_sbuf(col, fb))) break;
            const uint32_t kb = sKV + (uint32_t)st * p.stage_bytes;
            const uint32_t idS = ptx::idesc_bf16(BM, (uint32_t)cols, 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = ptx::sdesc_sw128(sQ + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
                const uint64_t b = ptx::sdesc_sw128(kb + (kk >> 2) * BN * 128 + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma(tmem + col, a, b, idS, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit(fb);
            ptx::tc_commit(bar(B_KV0 + kMaxStages + st));
            ++kv_it;
            if (j == J - 1) ptx::tc_commit(bar(B_Q_EMPTY));
            if (j >= 1) ok = issue_pv(j - 1, prev_cols);
            prev_cols = cols;
        }
        if (!ok) break;
        if (!(ok = issue_pv(J - 1, prev_cols))) break;
        if (AV) {
            uint32_t pb;
            if (!(ok = wait_p(pb))) break;
            if (!(ok = wait_bar(bar(B_AV_FULL), av_it & 1u, sh, p.err))) break;
            ++av_it;
            ptx::tc_fence_after();
            const uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
            const uint32_t pcol = TL::P + pb * (BN / 2);
            for (int kk = 0; kk < p.kpad_v / 16; ++kk) {
                const uint64_t b = ptx::sdesc_sw128(sAV + kk * 16 * 128, (uint32_t)p.kpad_v * 128, 1024);
                ptx::tc_mma_ts(tmem + TL::O, tmem + pcol + (uint32_t)(kk * 8), b, idPV, 1u);
            }
            ptx::tc_commit(bar(B_PV_DONE0 + (int)pb));
            ptx::tc_commit(bar(B_AV_EMPTY));
        }
        ptx::tc_commit(bar(B_O_FULL));
    }
    // every MMA issued by this thread completes before TMEM is released
    ptx::tc_commit(bar(B_DRAIN));
    drain_bar(bar(B_DRAIN), 0);
}

// ======================================================================= softmax / epilogue
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return ptx::pack_bf16x2(lo, hi); }

template <int D, bool AK, bool AV, bool T5, bool CAUSAL, int CPS>
__device__ void softmax_role(const Params &p, const Shared &sh, uint32_t tmem) {
    using TL = TmemLayout<CPS>;
    constexpr int BN = TL::BN;
    constexpr int NSPLIT = TL::NSPLIT;
    constexpr int NC = HC / KB;  // chunks per thread per key tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = (warp - TL::SW0) >> 2;    // which 64 keys of a key tile
    const int row = quad * 32 + lane;
    const int stid = threadIdx.x - 32 * TL::SW0;  // 0 .. 128*NSPLIT-1
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    float *Rrow = reinterpret_cast<float *>(sh.ptr + p.off_r) + row * p.SR;
    float *brow = reinterpret_cast<float *>(sh.ptr + p.off_beta) + row * p.SR;
    float *t5tab = reinterpret_cast<float *>(sh.ptr + p.off_t5);
    // exchange slots between the halves of a row: [parity][half][row] maxima, then
    // [half][row] x {l, low-bin sum, high-bin sum}
    float *xmax = reinterpret_cast<float *>(sh.ptr + p.off_x);
    float *xsum = xmax + 2 * 2 * BM;
    const float sl2 = p.scale_log2;
    const int k = p.clip_k;
    const int hi_off = CAUSAL ? 0 : k;  // largest offset held in the staged table rows
    const int W = p.W;
    uint32_t s_it = 0, p_item = 0, tiles = 0, grp = 0, pair_it = 0;
    const uint32_t gbar = bar(B_GROUP);
    const uint32_t pbar = bar(B_PAIR0 + quad);
    int t5_head = -1;
    bool ok = true;
    // tcgen05.ld/st are warp-collective (.sync.aligned): every decision guarding them is
    // uniform across the warp, and the warp reconverges before each TMEM access.
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = wait_bar(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    // the NSPLIT threads of the same rows (warps quad and quad + 4)
    auto pair_sync = [&]() -> bool {
        if (NSPLIT == 1) {
            __syncwarp();
            return true;
        }
        return group_sync(pbar, pair_it, sh, p.err);
    };
    // completion of the MMA that read P item `item` (each P buffer has its own barrier, and
    // that barrier cannot run two completions ahead: its next one needs our next item)
    auto wait_pv_item = [&](uint32_t item) -> bool {
        if (!wait_w(bar(B_PV_DONE0 + (int)(item & 1u)), (item >> 1) & 1u)) return false;
        ptx::tc_fence_after();
        __syncwarp();
        return true;
    };
    auto wait_sfull = [&](uint32_t &col, int &buf) -> bool {
        buf = (int)(s_it & 1u);
        if (!wait_w(bar(B_S_FULL0 + buf), (s_it >> 1) & 1u)) return false;
        ptx::tc_fence_after();
        __syncwarp();
        col = TL::S + (uint32_t)buf * BN;
        ++s_it;
        return true;
    };
    auto release_s = [&](int buf) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(B_S_EMPTY0 + buf));
    };

    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int bh, qt;
        decode_tile(p, t, bh, qt);
        const int i0 = qt * BM, gi = i0 + row, h = bh % p.H;
        const int gmin = i0 + quad * 32, gmax = gmin + 31;  // rows of this warp
        const int nk = keys_of(p, bh);
        const int nkc = tile_keys<CAUSAL>(p, bh, i0);
        const int J = (nkc + BN - 1) / BN;
        __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                              ((long long)bh * p.n + gi) * D;
        if (J == 0) {
            if (gi < p.n) {
#pragma unroll
                for (int c = 0; c < D / 8 / NSPLIT; ++c)
                    reinterpret_cast<uint4 *>(orow)[half * (D / 8 / NSPLIT) + c] = make_uint4(0, 0, 0, 0);
            }
            continue;
        }
        if (T5 && h != t5_head) {
            if (!(ok = group_sync(gbar, grp, sh, p.err))) break;
            for (int idx = stid; idx <= 2 * p.t5_R; idx += 128 * NSPLIT)
                t5tab[idx] = p.bias[t5_bucket(idx - p.t5_R, p.t5) * p.H + h] * kLog2e;
            if (!(ok = group_sync(gbar, grp, sh, p.err))) break;
            t5_head = h;
        }
        if (AK) {  // R row -> shared memory, split between the halves
            uint32_t col;
            int buf;
            if (!(ok = wait_sfull(col, buf))) break;
            for (int c0 = 16 * half; c0 < p.npad_k; c0 += 16 * NSPLIT) {
                uint32_t r[16];
                ptx::tmem_ld16(lane_base + col + (uint32_t)c0, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c0 + e < W) Rrow[c0 + e] = __uint_as_float(r[e]) * sl2;
            }
            release_s(buf);
        }
        if (AV && half == 0)
            for (int r = 0; r < W; ++r) brow[r] = 0.f;
        if (AK || AV) {
            if (!(ok = pair_sync())) break;  // R copied and bins cleared by both halves
        }
        float m_ref = -INFINITY, l = 0.f, lo_sum = 0.f, hi_sum = 0.f;

        for (int j = 0; j < J; ++j) {
            const int j0 = j * BN;
            const int cols = tile_cols<BN>(nkc, j);  // multiple of 32, > 0
            const int cbeg = half * NC;              // first chunk of this thread
            int live = cols / KB;                    // chunks any row of the warp can see
            if (CAUSAL) live = min(live, max(0, (gmax - j0) / KB + 1));
            uint32_t scol;
            int buf;
            if (!(ok = wait_sfull(scol, buf))) break;
            // ---- S chunks of this thread into registers
            float x[HC];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                if (cbeg + cc < live) {
                    __syncwarp();
                    ptx::tmem_ld32f(lane_base + scol + (uint32_t)((cbeg + cc) * KB), x + cc * KB);
                }
            }
            ptx::tmem_ld_wait();
            release_s(buf);
            // ---- logits in the log2 domain, relative term added, masks (S2-S4)
            float hmax = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                const int c = cbeg + cc;
                if (c >= live) continue;
                float *xc = x + cc * KB;
                const int e0 = j0 + c * KB;  // first key of the chunk
                // offsets j - i over the warp's rows lie in [e0 - gmax, e0 + 31 - gmin]
                const int lo_lim = T5 ? -p.t5_R : -k;      // at or below: first table row
                const int hi_lim = T5 ? p.t5_R : hi_off;   // at or above: last table row
                const bool w_left = (e0 + KB - 1 - gmin) <= lo_lim;
                const bool w_right = (e0 - gmax) >= hi_lim;
                const int base = e0 - gi;  // offset of element 0 for this row
                if (AK || T5) {
                    const float *tab = AK ? Rrow : t5tab;
                    const int lim = AK ? k : p.t5_R;
                    const int top = AK ? hi_off : p.t5_R;
                    if (w_left) {
                        const float cst = tab[0];
#pragma unroll
                        for (int e = 0; e < KB; ++e) xc[e] = fmaf(xc[e], sl2, cst);
                    } else if (w_right) {
                        const float cst = tab[lim + top];
#pragma unroll
                        for (int e = 0; e < KB; ++e) xc[e] = fmaf(xc[e], sl2, cst);
                    } else {
#pragma unroll
                        for (int e = 0; e < KB; ++e) {
                            const int o = min(top, max(-lim, base + e));
                            xc[e] = fmaf(xc[e], sl2, tab[o + lim]);
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < KB; ++e) xc[e] *= sl2;
                }
                const bool full = (e0 + KB <= nk) && (!CAUSAL || e0 + KB - 1 <= gmin);
                if (!full) {
#pragma unroll
                    for (int e = 0; e < KB; ++e) {
                        const int jj = e0 + e;
                        if (jj >= nk || (CAUSAL && jj > gi)) xc[e] = -INFINITY;
                    }
                }
#pragma unroll
                for (int e = 0; e < KB; ++e) hmax = fmaxf(hmax, xc[e]);
            }
            // ---- row maximum over both halves, lazy rescale (S5)
            float rmax = hmax;
            if (NSPLIT > 1) {
                float *slot = xmax + (j & 1) * 2 * BM;
                slot[half * BM + row] = hmax;
                if (!(ok = pair_sync())) break;
                rmax = fmaxf(hmax, slot[(1 - half) * BM + row]);
            }
            float alpha = 1.f;
            if (rmax > m_ref + kRescaleLog2) {
                alpha = ptx::ex2(m_ref - rmax);  // 0 while nothing was seen yet
                m_ref = rmax;
            }
            // on the first key tile l, the bins and O hold nothing yet: no rescale needed
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {  // same in every half
                l *= alpha;
                lo_sum *= alpha;
                hi_sum *= alpha;
                if (half == 0) {
                    if (AV && alpha != 1.f)
                        for (int r = 0; r < W; ++r) brow[r] *= alpha;
                    if (j >= 1) {  // O holds P V of the earlier key tiles
                        if (!(ok = wait_pv_item(p_item - 1))) break;
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t r[32];
                            ptx::tmem_ld32(lane_base + TL::O + (uint32_t)c0, r);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                            ptx::tmem_st32(lane_base + TL::O + (uint32_t)c0, r);
                        }
                        ptx::tmem_st_wait();
                    }
                }
                if (AV && NSPLIT > 1) {  // bins are rescaled before the other half adds new ones
                    if (!(ok = pair_sync())) break;
                }
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            // ---- exponentials, row sum, value bins (S7), P (bf16 pairs) into TMEM
            if (p_item >= 2) {  // the P buffer's previous P . V is done
                if (!(ok = wait_pv_item(p_item - 2))) break;
            }
            const uint32_t pbase = lane_base + TL::P + (p_item & 1u) * (BN / 2);
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                const int c = cbeg + cc;
                if (c * KB >= cols) continue;  // never read by P V
                const uint32_t pcol = pbase + (uint32_t)(c * (KB / 2));
                uint32_t pk[KB / 2];
                if (c >= live) {  // no row of this warp sees these keys
#pragma unroll
                    for (int e = 0; e < KB / 2; ++e) pk[e] = 0u;
                } else {
                    float *xc = x + cc * KB;
                    float rs = 0.f;
#pragma unroll
                    for (int e = 0; e < KB; ++e) {
                        xc[e] = ptx::ex2(xc[e] - m_use);
                        rs += xc[e];
                    }
                    l += rs;
                    if (AV) {
                        const int e0 = j0 + c * KB;
                        const bool w_left = (e0 + KB - 1 - gmin) <= -k;
                        const bool w_right = (e0 - gmax) >= hi_off;
                        if (w_left) {
                            lo_sum += rs;
                        } else if (w_right) {
                            hi_sum += rs;
                        } else {
                            // interior bins get exactly one key each over the whole row, so
                            // they are stored (not accumulated); the two end bins are sums
                            // branch-free: end-bin terms go to the sums, interior ones
                            // to their bin; the others write a spare slot (index W)
                            const int base = e0 - gi;
#pragma unroll
                            for (int e = 0; e < KB; ++e) {
                                const int o = base + e;
                                const bool lo = o <= -k, hi = !lo && o >= hi_off;
                                lo_sum += lo ? xc[e] : 0.f;
                                hi_sum += hi ? xc[e] : 0.f;
                                brow[(lo || hi) ? W : o + k] = xc[e];
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < KB / 2; ++e) pk[e] = pack2(xc[2 * e], xc[2 * e + 1]);
                }
                __syncwarp();
                ptx::tmem_st16(pcol, pk);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_P_FULL0 + (int)(p_item & 1u)));
            ++p_item;
        }
        if (!ok) break;
        // ---- combine the halves: l and the end-bin sums
        if (NSPLIT > 1) {
            xsum[(half * 3 + 0) * BM + row] = l;
            xsum[(half * 3 + 1) * BM + row] = lo_sum;
            xsum[(half * 3 + 2) * BM + row] = hi_sum;
            if (!(ok = pair_sync())) break;
            l += xsum[((1 - half) * 3 + 0) * BM + row];
            lo_sum += xsum[((1 - half) * 3 + 1) * BM + row];
            hi_sum += xsum[((1 - half) * 3 + 2) * BM + row];
        }
        if (AV) {
            // bins (bf16 pairs) become the A operand of O += beta W^V (written by half 0)
            if (p_item >= 2 && !(ok = wait_pv_item(p_item - 2))) break;
            if (half == 0) {
                brow[0] += lo_sum;
                brow[W - 1] += hi_sum;
                const uint32_t pbase = lane_base + TL::P + (p_item & 1u) * (BN / 2);
                for (int c0 = 0; c0 < p.kpad_v; c0 += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r0 = c0 + 2 * e;
                        pk[e] = pack2(r0 < W ? brow[r0] : 0.f, r0 + 1 < W ? brow[r0 + 1] : 0.f);
                    }
                    __syncwarp();
                    ptx::tmem_st16(pbase + (uint32_t)(c0 / 2), pk);
                }
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_P_FULL0 + (int)(p_item & 1u)));
            ++p_item;
        }
        // ---- epilogue (S8): O / l -> bf16 -> global, D / NSPLIT columns per thread
        if (!(ok = wait_w(bar(B_O_FULL), tiles & 1u))) break;
        ptx::tc_fence_after();
        __syncwarp();
        ++tiles;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c0 = half * (D / NSPLIT); c0 < (half + 1) * (D / NSPLIT); c0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld32(lane_base + TL::O + (uint32_t)c0, r);
            ptx::tmem_ld_wait();
            if (gi < p.n) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 v;
                    v.x = pack2(__uint_as_float(r[8 * q + 0]) * inv, __uint_as_float(r[8 * q + 1]) * inv);
                    v.y = pack2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv);
                    v.z = pack2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv);
                    v.w = pack2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv);
                    reinterpret_cast<uint4 *>(orow)[c0 / 8 + q] = v;
                }
            }
            __syncwarp();
        }
        ptx::tc_fence_before();
    }
}

// ======================================================================= kernel
template <int D, bool AK, bool AV, bool T5, bool CAUSAL, int CPS>
__global__ void __launch_bounds__(TmemLayout<CPS>::THREADS, CPS)
    relattn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kf,
                      const __grid_constant__ CUtensorMap tm_vf, const __grid_constant__ CUtensorMap tm_ak,
                      const __grid_constant__ CUtensorMap tm_av, const __grid_constant__ Params p) {
    using TL = TmemLayout<CPS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    Shared sh;
    sh.base = (raw + 1023u) & ~1023u;
    sh.ptr = smem_raw + (sh.base - raw);
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(sh.ptr + p.off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_ptr + kNumBars);
    sh.abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5;
    const uint32_t bars = sh.base + p.off_bar;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == B_S_EMPTY0 || i == B_S_EMPTY1 || i == B_P_FULL0 || i == B_P_FULL1 ||
                i == B_GROUP)
                cnt = 128 * TL::NSPLIT;
            if (i >= B_PAIR0 && i < B_PAIR0 + 4) cnt = 32 * TL::NSPLIT;
            ptx::mbar_init(bars + 8u * (uint32_t)i, cnt);
        }
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_kf);
        ptx::tma_prefetch_desc(&tm_vf);
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TL::cols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if ((threadIdx.x & 31) == 0) producer_role<D, AK, AV, CAUSAL, CPS>(p, sh, &tm_q, &tm_k, &tm_v, &tm_kf, &tm_vf, &tm_ak,
                                                      &tm_av);
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) mma_role<D, AK, AV, CAUSAL, CPS>(p, sh, tmem);
        __syncwarp();
    } else if (warp >= TL::SW0) {
        softmax_role<D, AK, AV, T5, CAUSAL, CPS>(p, sh, tmem);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TL::cols);
    }
}

}  // namespace tc
}  // namespace relattn
