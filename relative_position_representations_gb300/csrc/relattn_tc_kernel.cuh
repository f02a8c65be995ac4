// Fused relation-aware attention forward, bf16 in / fp32 accumulate, for sm_103a.
//
// Method: Shaw, Uszkoreit & Vaswani (paper summary page, section 3.4): eq. 4
//   e_ij = scale * (q_i . k_j + q_i . w^K_{clip(j-i,k)})        (the eq. 5 split)
// and eq. 3 split in two sums,
//   z_i = sum_j a_ij v_j + sum_r beta_ir w^V_r,   beta_ir = sum_{j: clip(j-i,k)+k = r} a_ij.
// T5 variant ("Relative position embeddings", section "T5"): e_ij = scale*q_i.k_j + b[bucket].
//
// One CTA per SM (persistent), looping over (query tile of 128 rows, head) work items,
// heaviest causal tiles first. Warp roles:
//   warp 0      TMA producer: Q tile + edge tables, then K/V tiles of 128 keys into a ring
//               of stages, in the order the MMA warp consumes them (K0 K1 V0 K2 V1 ...).
//   warp 1      MMA issuer (one thread): R = Q W^K^T once per tile (tiny N = table rows),
//               S_j = Q K_j^T into one of two TMEM score buffers, O += P_j V_j, and at the
//               end O += beta W^V. Accumulators live in TMEM (512 columns).
//   warps 2..5  softmax / epilogue, one thread per query row (TMEM lane): read S_j from TMEM,
//               add the gathered relative term (band tiles) or a per-row constant (tiles
//               entirely beyond +-k), mask, online softmax in the exp2 domain with a lazy
//               rescale (only when the row max grows by more than 2^8), write bf16 P to
//               shared memory, accumulate the 2k+1 value bins, then normalise O and store
//               it with TMA.
// Every wait is bounded; a wait that runs out sets the device status word and the CTA
// drains and exits.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "device_common.cuh"
#include "relattn_internal.h"
#include "sm103_ptx.cuh"

namespace relattn {
namespace tc {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // two score buffers: columns [0,128) and [128,256)
constexpr uint32_t kColO = 256;  // output accumulator: [256, 256+D)
constexpr uint32_t kColR = 384;  // relative-key products: [384, 384+npad_k), npad_k <= 128
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// barrier slots
enum : int {
    B_Q_FULL = 0, B_Q_EMPTY, B_S_FULL0, B_S_FULL1, B_S_EMPTY0, B_S_EMPTY1, B_P_FULL, B_PV_DONE,
    B_R_FULL, B_R_EMPTY, B_AV_FULL, B_AV_EMPTY, B_O_FULL, B_DRAIN, B_GROUP, B_KV0
};
constexpr int kMaxStages = 8;
constexpr int kNumBars = B_KV0 + 2 * kMaxStages;

struct Params {
    int BH, H, n;
    int n_qtiles, num_tiles;
    float scale_log2;   // scale * log2(e)
    const int *kv_len;  // [B] or null
    int *err;           // device status word
    int clip_k;         // Shaw: k
    int W;              // table rows staged: k+1 (causal) or 2k+1
    int SR;             // row stride (floats) of the per-row tables in shared memory
    int npad_k;         // W rounded up to 16: N of the R = Q W^K^T MMA
    int kpad_v;         // W rounded up to 16: K of the beta W^V MMA
    int table_heads;    // 1: tables indexed by head, 0: one shared table
    const float *bias;  // T5 [num_buckets, H]
    int t5_R;           // T5 offset-table radius (bucket is constant beyond it)
    T5Buckets t5;
    uint32_t off_q, off_kv, off_p, off_ak, off_av, off_r, off_beta, off_t5, off_bar;
    int stages;
    uint32_t stage_bytes;
};

struct Shared {
    uint32_t base;  // 1024-aligned shared address
    uint8_t *ptr;   // generic pointer to the same byte
    volatile int *abort_flag;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Shared &sh,
                                         int *err) {
    if (ptx::mbar_try(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try(bar, parity)) return true;
        if ((++spins & 127u) == 0) {
            if (*sh.abort_flag) return false;
            if (ptx::globaltimer() - t0 > kWaitLimitNs) {
                *sh.abort_flag = 1;
                atomicCAS(err, 0, 4 /* RELATTN_ERR_TIMEOUT */);
                return false;
            }
        }
    }
}

// Barrier among the 128 softmax threads, on an mbarrier so that the wait stays bounded
// (a plain bar.sync would hang if another thread of the group left after a timeout).
// The result is uniform across the calling warp.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t &it, const Shared &sh, int *err) {
    ptx::mbar_arrive(bar);
    const bool ok = wait_bar(bar, it & 1u, sh, err);
    ++it;
    return __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
}

__device__ __forceinline__ void decode_tile(const Params &p, int t, int &bh, int &qt) {
    qt = p.n_qtiles - 1 - t / p.BH;  // longest causal rows first
    bh = t % p.BH;
}

// number of allowed keys (before the causal clip) of the sequence of head bh
__device__ __forceinline__ int keys_of(const Params &p, int bh) {
    if (!p.kv_len) return p.n;
    return max(0, min(p.kv_len[bh / p.H], p.n));
}

template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles_of(const Params &p, int bh, int i0) {
    int nk = keys_of(p, bh);
    if (CAUSAL) nk = min(nk, i0 + BM);
    return (nk + BN - 1) / BN;
}

// ======================================================================= producer
template <int D, bool AK, bool AV, bool CAUSAL>
__device__ void producer_role(const Params &p, const Shared &sh, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                              const CUtensorMap *tm_ak, const CUtensorMap *tm_av) {
    constexpr int DB = D / 64;
    constexpr uint32_t kTileBytes = (uint32_t)BM * D * 2;
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
        const int J = kv_tiles_of<CAUSAL>(p, bh, i0);
        if (J == 0) continue;
        if (!(ok = wait_bar(bar(B_Q_EMPTY), (q_it & 1u) ^ 1u, sh, p.err))) break;
        const uint32_t qbytes = kTileBytes + (AK ? (uint32_t)p.npad_k * D * 2 : 0u);
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
            ptx::mbar_expect_tx(bar(B_KV0 + st), kTileBytes);
            const uint32_t dst = sKV + (uint32_t)st * p.stage_bytes;
#pragma unroll
            for (int blk = 0; blk < DB; ++blk)
                ptx::tma_load_3d(dst + blk * BN * 128, isK ? tm_k : tm_v, bar(B_KV0 + st),
                                 blk * 64, j * BN, bh);
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
        for (uint32_t it = kv_it > (uint32_t)S ? kv_it - S : 0; it < kv_it; ++it) {
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try(bar(B_KV0 + (int)(it % (uint32_t)S)), (it / (uint32_t)S) & 1u) &&
                   ptx::globaltimer() - t0 < kWaitLimitNs) {
            }
        }
        if (q_it) {
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try(bar(B_Q_FULL), (q_it - 1) & 1u) &&
                   ptx::globaltimer() - t0 < kWaitLimitNs) {
            }
        }
        if (AV && av_it) {
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try(bar(B_AV_FULL), (av_it - 1) & 1u) &&
                   ptx::globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ======================================================================= MMA issuer
template <int D, bool AK, bool AV, bool CAUSAL>
__device__ void mma_role(const Params &p, const Shared &sh, uint32_t tmem) {
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    const uint32_t sQ = sh.base + p.off_q, sKV = sh.base + p.off_kv, sP = sh.base + p.off_p;
    const uint32_t sAK = sh.base + p.off_ak, sAV = sh.base + p.off_av;
    const int S = p.stages;
    constexpr uint32_t idS = ptx::idesc_bf16(BM, BN, 0);
    constexpr uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
    const uint32_t idR = ptx::idesc_bf16(BM, (uint32_t)p.npad_k, 0);
    uint32_t kv_it = 0, q_it = 0, av_it = 0, s_it = 0, p_it = 0, tiles = 0;
    bool ok = true;

    // O += P_j V_j (P in shared memory, K-major; V tile MN-major)
    auto issue_pv = [&](int j) -> bool {
        if (!wait_bar(bar(B_P_FULL), p_it & 1u, sh, p.err)) return false;
        ++p_it;
        const int st = (int)(kv_it % (uint32_t)S);
        if (!wait_bar(bar(B_KV0 + st), (kv_it / (uint32_t)S) & 1u, sh, p.err)) return false;
        ptx::tc_fence_after();
        const uint32_t vb = sKV + (uint32_t)st * p.stage_bytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t a = ptx::sdesc_sw128(sP + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
            const uint64_t b = ptx::sdesc_sw128(vb + kk * 16 * 128, BN * 128, 1024);
            ptx::tc_mma(tmem + kColO, a, b, idPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::tc_commit(bar(B_PV_DONE));
        ptx::tc_commit(bar(B_KV0 + kMaxStages + st));
        ++kv_it;
        return true;
    };

    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int bh, qt;
        decode_tile(p, t, bh, qt);
        const int J = kv_tiles_of<CAUSAL>(p, bh, qt * BM);
        if (J == 0) continue;
        if (!(ok = wait_bar(bar(B_Q_FULL), q_it & 1u, sh, p.err))) break;
        ++q_it;
        ptx::tc_fence_after();
        if (AK) {
            if (!(ok = wait_bar(bar(B_R_EMPTY), (tiles & 1u) ^ 1u, sh, p.err))) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = ptx::sdesc_sw128(sQ + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
                const uint64_t b =
                    ptx::sdesc_sw128(sAK + (kk >> 2) * p.npad_k * 128 + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma(tmem + kColR, a, b, idR, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit(bar(B_R_FULL));
        }
        for (int j = 0; j < J && ok; ++j) {
            const int st = (int)(kv_it % (uint32_t)S);
            if (!(ok = wait_bar(bar(B_KV0 + st), (kv_it / (uint32_t)S) & 1u, sh, p.err))) break;
            const uint32_t buf = s_it & 1u;
            if (!(ok = wait_bar(bar(B_S_EMPTY0 + (int)buf), ((s_it >> 1) & 1u) ^ 1u, sh, p.err))) break;
            ptx::tc_fence_after();
            const uint32_t kb = sKV + (uint32_t)st * p.stage_bytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t a = ptx::sdesc_sw128(sQ + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
                const uint64_t b = ptx::sdesc_sw128(kb + (kk >> 2) * BN * 128 + (kk & 3) * 32, 16, 1024);
                ptx::tc_mma(tmem + kColS + buf * BN, a, b, idS, kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit(bar(B_S_FULL0 + (int)buf));
            ptx::tc_commit(bar(B_KV0 + kMaxStages + st));
            ++kv_it;
            ++s_it;
            if (j == J - 1) ptx::tc_commit(bar(B_Q_EMPTY));
            if (j >= 1) ok = issue_pv(j - 1);
        }
        if (!ok) break;
        if (!(ok = issue_pv(J - 1))) break;
        if (AV) {
            if (!(ok = wait_bar(bar(B_P_FULL), p_it & 1u, sh, p.err))) break;
            ++p_it;
            if (!(ok = wait_bar(bar(B_AV_FULL), av_it & 1u, sh, p.err))) break;
            ++av_it;
            ptx::tc_fence_after();
            for (int kk = 0; kk < p.kpad_v / 16; ++kk) {
                const uint64_t a = ptx::sdesc_sw128(sP + (kk >> 2) * BM * 128 + (kk & 3) * 32, 16, 1024);
                const uint64_t b = ptx::sdesc_sw128(sAV + kk * 16 * 128, (uint32_t)p.kpad_v * 128, 1024);
                ptx::tc_mma(tmem + kColO, a, b, idPV, 1u);
            }
            ptx::tc_commit(bar(B_AV_EMPTY));
        }
        ptx::tc_commit(bar(B_O_FULL));
        ++tiles;
    }
    // every MMA issued by this thread completes before TMEM is released
    ptx::tc_commit(bar(B_DRAIN));
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try(bar(B_DRAIN), 0) && ptx::globaltimer() - t0 < kWaitLimitNs) {
    }
}

// ======================================================================= softmax / epilogue
template <int D>
__device__ __forceinline__ bool store_tile(const Params &p, const Shared &sh, const CUtensorMap *tm_o,
                                           int i0, int bh, int stid, uint32_t &grp) {
    constexpr int DB = D / 64;
    const uint32_t gbar = sh.base + p.off_bar + 8u * B_GROUP;
    ptx::fence_proxy_async_smem();
    if (!group_sync(gbar, grp, sh, p.err)) return false;
    if (stid == 0) {
#pragma unroll
        for (int blk = 0; blk < DB; ++blk)
            ptx::tma_store_3d(tm_o, sh.base + p.off_p + blk * BM * 128, blk * 64, i0, bh);
        ptx::bulk_commit();
        ptx::bulk_wait_read0();
    }
    return group_sync(gbar, grp, sh, p.err);
}

// address of 16-byte chunk c (8 bf16 columns) of row `row` in a 128-byte-swizzled,
// K-major tile made of 64-column blocks of BM rows
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int row, int c) {
    return tile + (uint32_t)(c >> 3) * (BM * 128) + (uint32_t)row * 128 +
           (uint32_t)(((c & 7) ^ (row & 7)) << 4);
}

template <int D, bool AK, bool AV, bool T5, bool CAUSAL>
__device__ void softmax_role(const Params &p, const Shared &sh, uint32_t tmem,
                             const CUtensorMap *tm_o) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const int stid = threadIdx.x - 64;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    const uint32_t sP = sh.base + p.off_p;
    float *Rrow = reinterpret_cast<float *>(sh.ptr + p.off_r) + row * p.SR;
    float *brow = reinterpret_cast<float *>(sh.ptr + p.off_beta) + row * p.SR;
    float *t5tab = reinterpret_cast<float *>(sh.ptr + p.off_t5);
    const float sl2 = p.scale_log2;
    const int k = p.clip_k;
    const int hi_off = CAUSAL ? 0 : k;  // largest offset held in the staged table rows
    const int W = p.W;
    uint32_t s_it = 0, pv_base = 0, tiles = 0, grp = 0;
    const uint32_t gbar = bar(B_GROUP);
    int t5_head = -1;
    bool ok = true;
    // tcgen05.ld/st are warp-collective (.sync.aligned): every decision that guards them is
    // made uniform across the warp, and the warp reconverges before each TMEM access.
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = wait_bar(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };

    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        int bh, qt;
        decode_tile(p, t, bh, qt);
        const int i0 = qt * BM, gi = i0 + row, h = bh % p.H;
        const int nk = keys_of(p, bh);
        const int J = kv_tiles_of<CAUSAL>(p, bh, i0);
        if (J == 0) {
#pragma unroll
            for (int c = 0; c < D / 8; ++c) ptx::st_shared_v4(sw128_chunk(sP, row, c), 0, 0, 0, 0);
            ok = store_tile<D>(p, sh, tm_o, i0, bh, stid, grp);
            continue;
        }
        if (T5 && h != t5_head) {
            if (!(ok = group_sync(gbar, grp, sh, p.err))) break;
            for (int idx = stid; idx <= 2 * p.t5_R; idx += 128)
                t5tab[idx] = p.bias[t5_bucket(idx - p.t5_R, p.t5) * p.H + h] * kLog2e;
            if (!(ok = group_sync(gbar, grp, sh, p.err))) break;
            t5_head = h;
        }
        if (AK) {
            if (!(ok = wait_w(bar(B_R_FULL), tiles & 1u))) break;
            ptx::tc_fence_after();
            __syncwarp();
            for (int c0 = 0; c0 < p.npad_k; c0 += 16) {
                uint32_t r[16];
                ptx::tmem_ld16(lane_base + kColR + (uint32_t)c0, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c0 + e < W) Rrow[c0 + e] = __uint_as_float(r[e]) * sl2;
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_R_EMPTY));
        }
        if (AV)
            for (int r = 0; r < W; ++r) brow[r] = 0.f;
        float m_ref = -INFINITY, l = 0.f;

        for (int j = 0; j < J; ++j) {
            const uint32_t buf = s_it & 1u;
            if (!(ok = wait_w(bar(B_S_FULL0 + (int)buf), (s_it >> 1) & 1u))) break;
            ptx::tc_fence_after();
            __syncwarp();
            float s[BN];
            {
                uint32_t r[32];
#pragma unroll
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    ptx::tmem_ld32(lane_base + kColS + buf * BN + (uint32_t)c0, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[c0 + e] = __uint_as_float(r[e]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_S_EMPTY0 + (int)buf));
            ++s_it;

            const int j0 = j * BN;
            const int omin = j0 - (i0 + BM - 1), omax = j0 + BN - 1 - i0;  // offset range of the tile
            // ---- logits in the log2 domain, relative term added (S2-S4)
            if (AK) {
                if (omax <= -k) {
                    const float c = Rrow[0];
#pragma unroll
                    for (int e = 0; e < BN; ++e) s[e] = fmaf(s[e], sl2, c);
                } else if (omin >= hi_off) {
                    const float c = Rrow[W - 1];
#pragma unroll
                    for (int e = 0; e < BN; ++e) s[e] = fmaf(s[e], sl2, c);
                } else {
                    const int base = j0 - gi;
#pragma unroll
                    for (int e = 0; e < BN; ++e) {
                        const int o = min(hi_off, max(-k, base + e));
                        s[e] = fmaf(s[e], sl2, Rrow[o + k]);
                    }
                }
            } else if (T5) {
                const int R = p.t5_R;
                if (omax <= -R) {
                    const float c = t5tab[0];
#pragma unroll
                    for (int e = 0; e < BN; ++e) s[e] = fmaf(s[e], sl2, c);
                } else if (omin >= R) {
                    const float c = t5tab[2 * R];
#pragma unroll
                    for (int e = 0; e < BN; ++e) s[e] = fmaf(s[e], sl2, c);
                } else {
                    const int base = j0 - gi;
#pragma unroll
                    for (int e = 0; e < BN; ++e) {
                        const int o = min(R, max(-R, base + e));
                        s[e] = fmaf(s[e], sl2, t5tab[o + R]);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < BN; ++e) s[e] *= sl2;
            }
            // ---- masks: key padding and causal
            const bool full = (j0 + BN <= nk) && (!CAUSAL || j0 + BN - 1 <= i0);
            if (!full) {
#pragma unroll
                for (int e = 0; e < BN; ++e) {
                    const int jj = j0 + e;
                    if (jj >= nk || (CAUSAL && jj > gi)) s[e] = -INFINITY;
                }
            }
            // ---- online softmax (S5) with a lazy rescale
            float mx = s[0];
#pragma unroll
            for (int e = 1; e < BN; ++e) mx = fmaxf(mx, s[e]);
            const float m_new = fmaxf(m_ref, mx);
            float alpha = 1.f;
            if (m_new > m_ref + kRescaleLog2) {
                alpha = ptx::ex2(m_ref - m_new);
                m_ref = m_new;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            float rs = 0.f;
#pragma unroll
            for (int e = 0; e < BN; ++e) {
                s[e] = ptx::ex2(s[e] - m_use);
                rs += s[e];
            }
            l = l * alpha + rs;
            // ---- value bins (S7)
            if (AV) {
                if (alpha != 1.f)
                    for (int r = 0; r < W; ++r) brow[r] *= alpha;
                if (omax <= -k) {
                    brow[0] += rs;
                } else if (omin >= hi_off) {
                    brow[W - 1] += rs;
                } else {
                    const int base = j0 - gi;
#pragma unroll
                    for (int e = 0; e < BN; ++e) {
                        const int o = min(hi_off, max(-k, base + e));
                        brow[o + k] += s[e];
                    }
                }
            }
            // ---- the previous P.V must be done before P and O are touched
            if (j >= 1) {
                if (!(ok = wait_w(bar(B_PV_DONE), (pv_base + (uint32_t)j - 1u) & 1u))) break;
                ptx::tc_fence_after();
                // lanes that keep their max multiply by 1
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    __syncwarp();
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t r[32];
                        ptx::tmem_ld32(lane_base + kColO + (uint32_t)c0, r);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        ptx::tmem_st32(lane_base + kColO + (uint32_t)c0, r);
                    }
                    ptx::tmem_st_wait();
                }
            }
            // ---- P (bf16) to shared memory, 128-byte swizzled K-major
#pragma unroll
            for (int c = 0; c < BN / 8; ++c)
                ptx::st_shared_v4(sw128_chunk(sP, row, c), ptx::pack_bf16x2(s[8 * c], s[8 * c + 1]),
                                  ptx::pack_bf16x2(s[8 * c + 2], s[8 * c + 3]),
                                  ptx::pack_bf16x2(s[8 * c + 4], s[8 * c + 5]),
                                  ptx::pack_bf16x2(s[8 * c + 6], s[8 * c + 7]));
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_P_FULL));
        }
        if (!ok) break;
        if (AV) {
            // bins (bf16) become the A operand of O += beta W^V
            if (!(ok = wait_w(bar(B_PV_DONE), (pv_base + (uint32_t)J - 1u) & 1u))) break;
            for (int c = 0; c < p.kpad_v / 8; ++c) {
                float v8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v8[e] = (8 * c + e < W) ? brow[8 * c + e] : 0.f;
                ptx::st_shared_v4(sw128_chunk(sP, row, c), ptx::pack_bf16x2(v8[0], v8[1]),
                                  ptx::pack_bf16x2(v8[2], v8[3]), ptx::pack_bf16x2(v8[4], v8[5]),
                                  ptx::pack_bf16x2(v8[6], v8[7]));
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_P_FULL));
        }
        pv_base += (uint32_t)J;
        // ---- epilogue (S8): O / l -> bf16 -> TMA store
        if (!(ok = wait_w(bar(B_O_FULL), tiles & 1u))) break;
        ptx::tc_fence_after();
        __syncwarp();
        ++tiles;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld32(lane_base + kColO + (uint32_t)c0, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[8 * q + e]) * inv;
                ptx::st_shared_v4(sw128_chunk(sP, row, c0 / 8 + q), ptx::pack_bf16x2(f[0], f[1]),
                                  ptx::pack_bf16x2(f[2], f[3]), ptx::pack_bf16x2(f[4], f[5]),
                                  ptx::pack_bf16x2(f[6], f[7]));
            }
        }
        ptx::tc_fence_before();
        ok = store_tile<D>(p, sh, tm_o, i0, bh, stid, grp);
    }
    if (stid == 0) ptx::bulk_wait0();
}

// ======================================================================= kernel
template <int D, bool AK, bool AV, bool T5, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    relattn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ CUtensorMap tm_ak, const __grid_constant__ CUtensorMap tm_av,
                      const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
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
            if (i == B_S_EMPTY0 || i == B_S_EMPTY1 || i == B_P_FULL || i == B_R_EMPTY ||
                i == B_GROUP)
                cnt = 128;
            ptx::mbar_init(bars + 8u * (uint32_t)i, cnt);
        }
        *sh.abort_flag = 0;
        ptx::mbar_init_fence();
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_o);
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if ((threadIdx.x & 31) == 0) producer_role<D, AK, AV, CAUSAL>(p, sh, &tm_q, &tm_k, &tm_v, &tm_ak, &tm_av);
        __syncwarp();
    } else if (warp == 1) {
        if ((threadIdx.x & 31) == 0) mma_role<D, AK, AV, CAUSAL>(p, sh, tmem);
        __syncwarp();
    } else {
        softmax_role<D, AK, AV, T5, CAUSAL>(p, sh, tmem, &tm_o);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace tc
}  // namespace relattn
