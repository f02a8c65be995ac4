// Fused relation-aware attention forward, bf16 in / fp32 accumulate, for sm_103a.
//
// Method: Shaw, Uszkoreit & Vaswani (paper summary page, section 3.4): eq. 4 in the split
// form of eq. 5,
//   e_ij = scale * (q_i . k_j + R_i[clip(j-i,k)+k]),    R = Q W^K^T  ([BM x (2k+1)] per tile),
// and eq. 3 split in two sums,
//   z_i = sum_j a_ij v_j + sum_r beta_ir w^V_r,   beta_ir = sum_{j: clip(j-i,k)+k = r} a_ij.
// Scalar-bias variant ("Relative position embeddings", sections "T5" and "Placement in the
// taxonomy"): e_ij = scale*q_i.k_j + b_h(j - i), with b a T5 bucket's table entry, ALiBi's
// -m_h |j - i|, or a per-offset table clipped at its radius; the kernel reads b from a
// shared-memory table over the offsets (constant beyond its radius).
//
// One persistent CTA per SM. A work item is two query tiles of 128 rows ("slots" 0 and 1):
// normally two neighbouring tiles of the same head, which then share every K/V tile, or,
// for heads with an odd number of query tiles, the leftover tiles of two heads. Items are
// scheduled in groups of heads whose K/V fit in half of L2, longest causal rows first. When
// the per-row tables of two slots do not fit shared memory, an item is one tile.
// Warp roles (384 threads):
//   warp 0      TMA producer (the whole warp runs it, one elected lane issues): both Q tiles
//               and the edge tables, then K/V tiles of 128 keys
//               (whole-tile boxes, 32-row boxes for the last, partly valid tile) into a ring,
//               in the order the MMA warp consumes them.
//   warps 1-2   MMA issuers, one per slot (the whole warp runs it; one elected lane issues
//               each tcgen05 instruction, so operands stay warp-uniform): R = Q W^K^T,
//               S_j = Q K_j^T, O += P_j V_j (P read from TMEM), O += beta W^V, walking the
//               K/V ring in the order it was filled; the two slots' chains run side by side.
//   warp 3      idle (registers are allocated per 4-warp group).
//   warps 4-7   softmax / epilogue of slot 0, warps 8-11 of slot 1: one thread per query row
//               (= TMEM lane) holding the whole 128-key score row. The relative term is a
//               per-row constant on 32-key chunks that lie beyond +-k for the whole warp (the
//               scale and that constant then fold into the exponent's FMA, and the row
//               maximum is taken on the raw scores) and a shared-memory gather inside the
//               band; online softmax in the exp2 domain with a lazy rescale (only when the
//               running max grows by more than 2^8); value bins; bf16 P into TMEM; epilogue
//               O / l -> bf16 -> global.
// TMEM (512 columns): S of slot s at 128 s, O at 256 + D s; P (bf16 pairs, 64 columns) at
// 384 + 64 s when D = 64, over the first half of the slot's S when D = 128. With its own P
// columns a slot's S_{j+1} is computed while its softmax still works on S_j; over S, S_{j+1}
// waits for the P_j . V_j that reads those columns.
// Every wait is bounded; a wait that runs out sets the device status word and the CTA drains
// and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "relattn_internal.h"
#include "sm103_ptx.cuh"

namespace relattn {
namespace tc {

constexpr int BM = 128;        // query rows per tile (= TMEM lanes)
constexpr int BN = 128;        // keys per key tile
constexpr int KB = 32;         // key rows per partial TMA box and keys per softmax chunk
constexpr int NCH = BN / KB;   // chunks per key tile
constexpr int kThreads = 384;
constexpr int kSoftWarp0 = 4;  // first softmax warp; slot s uses warps 4 + 4 s .. 7 + 4 s
// registers per thread: launched with kLaunchRegs; the producer/MMA warpgroup hands
// registers to the two softmax warpgroups (sum stays kThreads * kLaunchRegs)
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 72;
constexpr int kSoftRegs = 216;
static_assert(128 * kCtrlRegs + 256 * kSoftRegs == kThreads * kLaunchRegs, "register split");
static_assert(BM == 128 && BN == 128, "the MMA chains (ptx::tc_mma_*_k*) assume 128-row operand tiles");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
// Every device wait is bounded by Params::wait_limit SM clock cycles (the library default
// is 2e9, about one second at 2 GHz); clock64 is read only after a wait did not succeed at
// once and then every 256 polls.

// TMEM columns of slot s. D = 64: S at 128 s, O at 256 + 64 s, P at 384 + 64 s. D = 128 with
// two tiles per item: S at 128 s, O at 256 + 128 s, P over the first half of the slot's S.
// D = 128 with one tile per item (SG): S at 0, O at 128, P at 256.
template <int D, bool SG>
struct Tm {
    static constexpr bool P_ALIAS = D == 128 && !SG;
    static __device__ __forceinline__ uint32_t S(int s) { return (SG && D == 128) ? 0u : 128u * (uint32_t)s; }
    static __device__ __forceinline__ uint32_t O(int s) {
        return (SG && D == 128) ? 128u : 256u + (uint32_t)(D * s);
    }
    static __device__ __forceinline__ uint32_t P(int s) {
        if (SG && D == 128) return 256u;
        return P_ALIAS ? 128u * (uint32_t)s : 384u + 64u * (uint32_t)s;
    }
    // value bins (bf16 pairs, up to 64 columns): the upper half of the slot's S columns, which
    // hold nothing live once the item's last score tile is in registers (P over S takes only
    // the lower half), so the bins never wait for the last P . V
    static __device__ __forceinline__ uint32_t Bn(int s) { return S(s) + 64u; }
};

// barrier slots
enum : int {
    SB_S_FULL = 0, SB_S_EMPTY, SB_P_FULL, SB_PV_DONE, SB_O_FULL, SB_DRAIN, SB_BN_FULL, SB_BN_DONE,
    SB_Q_FULL, SB_Q_EMPTY, SB_AV_FULL, SB_AV_EMPTY,  // split feed only
    kSlotBars
};
enum : int {
    B_Q_FULL = 0, B_Q_EMPTY, B_AV_FULL, B_AV_EMPTY, B_UNUSED,  // shared feed only
    B_SLOT0 = 5,  // per slot: the SB_* barriers
    B_KV0 = B_SLOT0 + 2 * kSlotBars
};
constexpr int kMaxStages = 8;
constexpr int kNumBars = B_KV0 + 2 * kMaxStages;

struct Params {
    int BH, H, n;
    int n_qtiles, num_items, head_group;
    int items_full, n_groups;  // items of a whole head group; head groups (the last may be short)
    int rot_step;              // items_full mod the grid size
    int tail_from;             // first item of the split last wave (num_items if none)
    int snake;                 // items differ in length: alternate the wave direction
    uint32_t off_list;         // shared-memory offset of the snake-order item list
    float scale_log2;   // scale * log2(e)
    const int *kv_len;  // [B] or null
    int *err;           // device status word
    void *out;          // [B, H, n, D] bf16
    int clip_k;         // Shaw: k
    int W;              // table rows staged: k+1 (causal) or 2k+1
    int SR;             // row stride (floats) of the R rows in shared memory
    int SB;             // row stride (floats) of the value bins, with a spare slot at index W
    int pair;           // 1: two query tiles per item, 0: one
    int npad_k;         // W rounded up to 16: N of the R = Q W^K^T MMA
    int kpad_v;         // W rounded up to 16: K of the beta W^V MMA
    int table_heads;    // 1: tables indexed by head, 0: one shared table
    int two_tables;     // the two slots may belong to different heads: own table buffers
    const float *bias;  // scalar bias: T5 [num_buckets, H], ALiBi slopes [H] or [H|1, 2R+1]
    int bias_kind;      // BiasKind
    int bias_R;         // kBiasTable: the table's clip radius
    long long bias_hs;  // kBiasTable: head stride of the table (0 = shared)
    int t5_R;           // offset-table radius (the bias is constant beyond it)
    T5Buckets t5;
    uint32_t off_q[2], off_kv, off_ak[2], off_av[2], off_r[2], off_beta[2], off_t5[2], off_bar;
    // Two ways to feed the slots. Shared: one producer warp, one K/V ring whose entries may
    // serve both slots (two query tiles of one head share K/V), and one Q and one W^V barrier
    // pair for both. Split (items of two one-tile heads, nothing to share): each slot has its
    // own producer warp, its own half of the ring and its own Q and W^V barriers, so the two
    // slots run their items independently.
    int split;
    long long wait_limit;  // bound of every wait, SM clock cycles
    int withhold_q;        // test hook: the producer issues no Q load for its first item
    int stages;
    int ring_stages;     // stages of one ring: all of them (shared feed) or half (split feed)
    uint32_t stage_bytes;
    uint32_t stage_mul;  // ceil(2^32 / ring_stages): e / ring_stages = umulhi(e, stage_mul)
                         // for the ring positions used (e < 2^29)
};

// ring position e -> (stage within the ring, round) without a division
__device__ __forceinline__ void ring_pos(const Params &p, uint32_t e, uint32_t &stage, uint32_t &round) {
    round = __umulhi(e, p.stage_mul);
    stage = e - round * (uint32_t)p.ring_stages;
}

struct Shared {
    uint32_t base;  // 1024-aligned shared address
    uint8_t *ptr;   // generic pointer to the same byte
    volatile int *abort_flag;
    long long limit;  // bound of every wait (cycles)
};

// slow path of a bounded wait (polls, with an abort check and a cycle limit every 256 polls)
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           int *err, long long limit) {
    const long long t0 = clock64();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try(bar, parity)) return true;
        if ((++spins & 255u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(err, 0, 4 /* RELATTN_ERR_TIMEOUT */);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Shared &sh,
                                         int *err) {
    if (ptx::mbar_try(bar, parity)) return true;
    return wait_bar_slow(bar, parity, sh.abort_flag, err, sh.limit);
}

// the same for the producer and MMA warps, with the slow path out of line (those warps have
// registers to spare for a call, and their many waits would otherwise each carry a copy)
static __device__ __noinline__ bool wait_bar_slow_call(uint32_t bar, uint32_t parity,
                                                volatile int *abort_flag, int *err,
                                                long long limit) {
    return wait_bar_slow(bar, parity, abort_flag, err, limit);
}
__device__ __forceinline__ bool wait_bar_ctrl(uint32_t bar, uint32_t parity, const Shared &sh,
                                              int *err) {
    if (ptx::mbar_try(bar, parity)) return true;
    return wait_bar_slow_call(bar, parity, sh.abort_flag, err, sh.limit);
}

// bounded poll of a barrier during teardown (no abort check)
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!ptx::mbar_try(bar, parity) && clock64() - t0 < limit) {
    }
}

// Barrier among the 128 softmax threads of a slot (hardware named barrier 1 + slot): warps
// blocked in it take no issue slots. `ok` is AND-reduced over the 128 threads, so every
// thread sees the same result; all 128 threads always reach it together (they follow the
// same item / tile sequence and leave it at the same point), so it cannot hang.
__device__ __forceinline__ bool slot_sync(int slot, bool ok) {
    return ptx::bar_red_and(1 + slot, 128, ok);
}

// ----------------------------------------------------------------------- work items
struct Item {
    int bh[2], qt[2];
    bool valid[2];
    bool shared;  // both slots are tiles of one head: they share K/V
};

__host__ __device__ inline int items_per_group(int gsize, int Q, int pair) {
    if (!pair) return Q * gsize;
    return ((Q & 1) ? (gsize + 1) / 2 : 0) + (Q >> 1) * gsize;
}

// Items of a group of heads: first the leftover (last, longest) query tile of heads with an
// odd tile count, two heads per item; then pairs (2i+1, 2i) of the same head, i descending.
// Without pairing an item is one tile, again longest first.
__device__ __forceinline__ Item decode_pair_item(const Params &p, int t) {
    const int Q = p.n_qtiles, G = p.head_group;
    const int full = items_per_group(G, Q, p.pair);
    const int g = t / full;
    int r = t - g * full;
    const int g0 = g * G;
    const int gsize = min(G, p.BH - g0);
    Item it;
    if (!p.pair) {
        it.qt[0] = it.qt[1] = Q - 1 - r / gsize;
        it.bh[0] = it.bh[1] = g0 + r % gsize;
        it.valid[0] = true;
        it.valid[1] = false;
        it.shared = false;
        return it;
    }
    const int singles = (Q & 1) ? (gsize + 1) / 2 : 0;
    if (r < singles) {
        it.qt[0] = it.qt[1] = Q - 1;
        it.bh[0] = g0 + 2 * r;
        it.bh[1] = g0 + 2 * r + 1;
        it.valid[0] = true;
        it.valid[1] = 2 * r + 1 < gsize;
        it.shared = false;
    } else {
        r -= singles;
        const int i = (Q >> 1) - 1 - r / gsize;
        const int h = g0 + r % gsize;
        it.bh[0] = it.bh[1] = h;
        it.qt[0] = 2 * i + 1;
        it.qt[1] = 2 * i;
        it.valid[0] = it.valid[1] = true;
        it.shared = true;
    }
    return it;
}

// Item t of the launch. Items from tail_from on split the last, partial wave of two-tile
// items into one-tile items (the pair item tail_from + u / 2 gives its tile u % 2, run in
// slot 0), so that wave costs about half a two-tile item on twice as many CTAs.
__device__ __forceinline__ Item decode_item(const Params &p, int t) {
    int single = -1;
    if (t >= p.tail_from) {
        const int u = t - p.tail_from;
        t = p.tail_from + (u >> 1);
        single = u & 1;
    }
    Item it = decode_pair_item(p, t);
    if (single >= 0) {
        if (single == 1) {
            it.bh[0] = it.bh[1];
            it.qt[0] = it.qt[1];
            it.valid[0] = it.valid[1];
        }
        it.valid[1] = false;
        it.shared = false;
    }
    return it;
}

// number of allowed keys (before the causal clip) of the sequence of head bh
__device__ __forceinline__ int keys_of(const Params &p, int bh) {
    if (!p.kv_len) return p.n;
    return max(0, min(p.kv_len[bh / p.H], p.n));
}

// Work order of a CTA. A head group's items come longest first (decode_item). Items of one
// length (snake = 0): CTA b takes items b, b + gridDim.x, ... Items that differ in length
// (causal query tiles of long sequences): the CTAs take a group's items in waves of gridDim.x
// whose direction alternates from wave to wave, so that a CTA that took one of the longest
// items of a wave takes one of the shortest of the next, and group g's waves start rotated
// by g * (items per group mod gridDim.x), so that the partial last waves of successive groups
// land on different CTAs. Every role of a CTA walks the same order.
constexpr int kListCap = 256;  // entries of the shared-memory item list (snake order)
// Padding of the offset-bias table on each side: a banded chunk of a warp reaches at most 61
// offsets beyond the table's ends (31 rows of the warp + 30 keys of the chunk)
constexpr int kT5Pad = 64;

// The snake order of this CTA, written once by one thread before the roles start (into a
// list of kListCap entries ending in -1; the host enables the order only when it fits).
__device__ __forceinline__ void snake_list(const Params &p, int *list) {
    const int G = (int)gridDim.x;
    int n = 0;
    for (int g = 0; g < p.n_groups; ++g) {
        const int cnt = g + 1 < p.n_groups ? p.items_full : p.num_items - g * p.items_full;
        int bg = (int)blockIdx.x - (g * p.rot_step) % G;
        if (bg < 0) bg += G;
        // a position past the group's end stays past it in later waves
        for (int k = 0;; ++k) {
            const int r = k * G + ((k & 1) ? G - 1 - bg : bg);
            if (r >= cnt || n + 1 >= kListCap) break;
            list[n++] = g * p.items_full + r;
        }
    }
    list[n] = -1;
}
struct Sched {
    int i;            // items taken so far
    const int *list;  // the snake order, or null for CTA b taking b, b + gridDim.x, ...
    __device__ __forceinline__ Sched(const Params &p, const Shared &sh)
        : i(0), list(p.snake ? reinterpret_cast<const int *>(sh.ptr + p.off_list) : nullptr) {}
    __device__ __forceinline__ int next(const Params &p) {
        if (list) return list[i++];
        const int t = (int)blockIdx.x + i * (int)gridDim.x;
        ++i;
        return t < p.num_items ? t : -1;
    }
};

// one slot's share of item t: head, query tile and the allowed keys of that head; not valid
// past the last item (t < 0 or t >= num_items) or when the slot has no tile in it
struct SlotItem {
    int bh, qt, nk;
    bool valid;
};
__device__ __forceinline__ SlotItem slot_item(const Params &p, int t, int slot) {
    SlotItem r{0, 0, 0, false};
    if (t >= 0 && t < p.num_items) {
        const Item it = decode_item(p, t);
        r.valid = it.valid[slot];
        r.bh = it.bh[slot];
        r.qt = it.qt[slot];
        if (r.valid) r.nk = keys_of(p, r.bh);
    }
    return r;
}

// keys any row of query tile qt may see
template <bool CAUSAL>
__device__ __forceinline__ int tile_keys(const Params &p, int bh, int qt) {
    const int nk = keys_of(p, bh);
    return CAUSAL ? min(nk, qt * BM + BM) : nk;
}

// columns of key tile j that are loaded and multiplied: the allowed keys rounded up to
// whole 32-row boxes
__device__ __forceinline__ int tile_cols(int nkc, int j) {
    const int c = nkc - j * BN;
    return c >= BN ? BN : ((c + KB - 1) / KB) * KB;
}

// K/V ring order of an item, which is also the order the MMA warp consumes the entries in.
// Every slot starts with K_0. With its own P columns (EARLY_S) a slot then takes K_{j+1}
// before V_j, so S_{j+1} is computed while its softmax works on S_j; with P over S it takes
// V_j before K_{j+1}. Shared items hold one entry per tile for both slots (an entry serves
// every slot whose tiles reach it); otherwise each slot has its own entries, interleaved.
template <bool CAUSAL, bool EARLY_S>
struct Plan {
    int nkc[2], J[2];
    int Jmax;
    bool shared;
    __device__ __forceinline__ void make(const Params &p, const Item &it) {
        shared = it.shared;
        Jmax = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            nkc[s] = it.valid[s] ? tile_keys<CAUSAL>(p, it.bh[s], it.qt[s]) : 0;
            J[s] = (nkc[s] + BN - 1) / BN;
            Jmax = max(Jmax, J[s]);
        }
    }
    __device__ __forceinline__ bool active(int s) const { return J[s] > 0; }
    // split feed: the plan of slot s alone (the other slot's tiles come from its own ring)
    __device__ __forceinline__ void keep_only(int s) {
        J[1 - s] = 0;
        nkc[1 - s] = 0;
        shared = false;
        Jmax = J[s];
    }
    // slots (bit mask) that use K or V tile j
    __device__ __forceinline__ int users(int j) const {
        return (j < J[0] ? 1 : 0) | (j < J[1] ? 2 : 0);
    }
    // The entries come in groups: group 0 is K_0; then, per tile j, the groups K_{j+1} and
    // V_j (in the order above). A group is one entry in shared items and one entry per slot
    // that has that tile otherwise. Callers walk g = 0 .. groups()-1 and e = 0 .. 1 with
    // entry(g, e, ...), so the per-entry code exists once.
    __device__ __forceinline__ int groups() const { return 1 + 2 * Jmax; }
    // entry e of group g: false if there is none; else isK, tile j, slot mask and source slot
    __device__ __forceinline__ bool entry(int g, int e, bool &isK, int &j, int &mask, int &src) const {
        if (g == 0) {
            isK = true;
            j = 0;
        } else {
            const int jj = (g - 1) >> 1;
            const bool first = ((g - 1) & 1) == 0;
            isK = EARLY_S ? first : !first;
            j = isK ? jj + 1 : jj;
        }
        if (shared) {
            src = 0;
            mask = e == 0 ? users(j) : 0;
        } else {
            src = e;
            mask = j < J[e] ? (1 << e) : 0;
        }
        return mask != 0;
    }
    // keys of tile j loaded for an entry (the largest of the slots using it)
    __device__ __forceinline__ int load_cols(int j, int mask) const {
        int c = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s)
            if (mask & (1 << s)) c = max(c, tile_cols(nkc[s], j));
        return c;
    }
};

// ======================================================================= producer
// Shared feed: one warp loads for both slots. Split feed: warp `me` loads for slot `me` only,
// into its own ring (stages ring0 .. ring0 + ring_stages - 1) and on the slot's own barriers.
template <int D, bool SG, bool AK, bool AV, bool CAUSAL>
__device__ void producer_role(const Params &p, const Shared &sh, const CUtensorMap *tm_q,
                              const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                              const CUtensorMap *tm_kf, const CUtensorMap *tm_vf,
                              const CUtensorMap *tm_ak, const CUtensorMap *tm_av, int me_in) {
    constexpr int DB = D / 64;
    constexpr bool EARLY_S = !Tm<D, SG>::P_ALIAS;
    const bool SPLIT = p.split != 0;
    const int me = __shfl_sync(0xffffffffu, me_in, 0);
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    auto sbar = [&](int s, int which) { return bar(B_SLOT0 + kSlotBars * s + which); };
    const uint32_t q_full = SPLIT ? sbar(me, SB_Q_FULL) : bar(B_Q_FULL);
    const uint32_t q_empty = SPLIT ? sbar(me, SB_Q_EMPTY) : bar(B_Q_EMPTY);
    const uint32_t av_full = SPLIT ? sbar(me, SB_AV_FULL) : bar(B_AV_FULL);
    const uint32_t av_empty = SPLIT ? sbar(me, SB_AV_EMPTY) : bar(B_AV_EMPTY);
    const int ring0 = SPLIT ? me * p.ring_stages : 0;
    const uint32_t sKV = sh.base + p.off_kv;
    const int S = p.ring_stages;
    // the whole warp runs this role; waits are made warp-uniform and one lane issues
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    uint32_t kv_it = 0, q_it = 0, av_it = 0;
    bool ok = true;
    Sched sc(p, sh);
    for (int t = sc.next(p); t >= 0 && ok; t = sc.next(p)) {
        const Item it = decode_item(p, t);
        Plan<CAUSAL, EARLY_S> pl;
        pl.make(p, it);
        if (SPLIT) pl.keep_only(me);
        if (pl.Jmax == 0) continue;
        if (!(ok = wait(q_empty, (q_it & 1u) ^ 1u))) break;
        ++q_it;
        // edge-table buffer b serves slot b (two_tables) or both slots; tab_head[b] < 0: unused
        int tab_head[2] = {-1, -1};
        if (SPLIT) {  // own buffers (two_tables is set with the split feed)
            tab_head[me] = p.table_heads ? it.bh[me] % p.H : 0;
        } else if (p.two_tables) {
            for (int s = 0; s < 2; ++s)
                if (pl.active(s)) tab_head[s] = p.table_heads ? it.bh[s] % p.H : 0;
        } else {
            const int s = pl.active(0) ? 0 : 1;
            tab_head[0] = p.table_heads ? it.bh[s] % p.H : 0;
        }
        uint32_t qbytes = 0;
        for (int s = 0; s < 2; ++s) {
            if (pl.active(s)) qbytes += (uint32_t)BM * D * 2;
            if (AK && tab_head[s] >= 0) qbytes += (uint32_t)p.npad_k * D * 2;
        }
        ptx::mbar_expect_tx_w(q_full, qbytes);
        // test hook: the first item's Q tiles are announced but never loaded, so the MMA warp's
        // bounded wait for them runs out (the device status word reports the timeout)
        const bool hold = p.withhold_q && q_it == 1;
        for (int s = 0; s < 2; ++s) {
            if (pl.active(s) && !hold) {
                const uint32_t sQ = sh.base + p.off_q[s];
#pragma unroll
                for (int blk = 0; blk < DB; ++blk)
                    ptx::tma_load_3d_w(sQ + blk * BM * 128, tm_q, q_full, blk * 64,
                                     it.qt[s] * BM, it.bh[s]);
            }
            if (AK && tab_head[s] >= 0) {
                const uint32_t sAK = sh.base + p.off_ak[s];
#pragma unroll
                for (int blk = 0; blk < DB; ++blk)
                    ptx::tma_load_3d_w(sAK + blk * p.npad_k * 128, tm_ak, q_full, blk * 64, 0,
                                     tab_head[s]);
            }
        }
        for (int g = 0; g < pl.groups() && ok; ++g) {
            for (int e = 0; e < 2; ++e) {
                bool isK;
                int j, mask, src;
                if (!pl.entry(g, e, isK, j, mask, src)) continue;
                uint32_t st_u, round;
                ring_pos(p, kv_it, st_u, round);
                const int st = ring0 + (int)st_u;
                if (!(ok = wait(bar(B_KV0 + kMaxStages + st), (round & 1u) ^ 1u))) break;
                const int nbox = pl.load_cols(j, mask) / KB;
                ptx::mbar_expect_tx_w(bar(B_KV0 + st), (uint32_t)nbox * KB * D * 2);
                const uint32_t dst = sKV + (uint32_t)st * p.stage_bytes;
                const int bh = it.bh[src];
                if (nbox == BN / KB) {  // whole tile: one box of 128 rows per 64-column block
#pragma unroll
                    for (int blk = 0; blk < DB; ++blk)
                        ptx::tma_load_3d_w(dst + blk * BN * 128, isK ? tm_kf : tm_vf, bar(B_KV0 + st),
                                         blk * 64, j * BN, bh);
                } else {  // last tile: only the 32-row boxes holding allowed keys
                    for (int b = 0; b < nbox; ++b) {
#pragma unroll
                        for (int blk = 0; blk < DB; ++blk)
                            ptx::tma_load_3d_w(dst + blk * BN * 128 + b * KB * 128, isK ? tm_k : tm_v,
                                             bar(B_KV0 + st), blk * 64, j * BN + b * KB, bh);
                    }
                }
                ++kv_it;
            }
        }
        if (!ok) break;
        if (AV) {
            if (!(ok = wait(av_empty, (av_it & 1u) ^ 1u))) break;
            ++av_it;
            uint32_t vbytes = 0;
            for (int s = 0; s < 2; ++s)
                if (tab_head[s] >= 0) vbytes += (uint32_t)p.kpad_v * D * 2;
            ptx::mbar_expect_tx_w(av_full, vbytes);
            for (int s = 0; s < 2; ++s) {
                if (tab_head[s] < 0) continue;
                const uint32_t sAV = sh.base + p.off_av[s];
#pragma unroll
                for (int blk = 0; blk < DB; ++blk)
                    ptx::tma_load_3d_w(sAV + blk * p.kpad_v * 128, tm_av, av_full, blk * 64, 0,
                                     tab_head[s]);
            }
        }
    }
    // drain: wait (bounded) for the copies issued into shared memory, so that none is still
    // in flight when the CTA exits (normally they were all consumed already; after an abort
    // the consumers may have given up on some)
    for (uint32_t i = kv_it > (uint32_t)S ? kv_it - S : 0; i < kv_it; ++i) {
        uint32_t st_u, round;
        ring_pos(p, i, st_u, round);
        drain_bar(bar(B_KV0 + ring0 + (int)st_u), round & 1u, sh.limit);
    }
    if (q_it) drain_bar(q_full, (q_it - 1) & 1u, sh.limit);
    if (AV && av_it) drain_bar(av_full, (av_it - 1) & 1u, sh.limit);
}

// ======================================================================= MMA issuers
// One MMA warp per slot (warps 1 and 2), so the two slots' wait-issue-commit chains run side
// by side. Shared feed: both warps walk every item's K/V ring entries in ring order and each
// releases every entry (a tcgen05 commit after its MMAs on it, or a plain arrive when its
// slot does not use it): the release barriers count two arrivals. A warp releases an entry,
// Q or the W^V rows only after waiting for them to be filled, so neither warp can arrive for
// a later fill than the producer has made. Split feed: each warp walks its own slot's ring
// and barriers, which count one arrival. The whole warp runs the role with warp-uniform
// control flow; one elected lane issues each tcgen05 instruction.
template <int D, bool SG, bool AK, bool AV, bool CAUSAL>
__device__ void mma_role(const Params &p, const Shared &sh, uint32_t tmem, int slot_in) {
    using T = Tm<D, SG>;
    const int slot = __shfl_sync(0xffffffffu, slot_in, 0);  // known warp-uniform from here on
    constexpr bool EARLY_S = !T::P_ALIAS;
    const bool SPLIT = p.split != 0;
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    auto sbar = [&](int which) { return bar(B_SLOT0 + kSlotBars * slot + which); };
    const uint32_t q_full = SPLIT ? sbar(SB_Q_FULL) : bar(B_Q_FULL);
    const uint32_t q_empty = SPLIT ? sbar(SB_Q_EMPTY) : bar(B_Q_EMPTY);
    const uint32_t av_full = SPLIT ? sbar(SB_AV_FULL) : bar(B_AV_FULL);
    const uint32_t av_empty = SPLIT ? sbar(SB_AV_EMPTY) : bar(B_AV_EMPTY);
    const int ring0 = SPLIT ? slot * p.ring_stages : 0;
    constexpr uint32_t idPV = ptx::idesc_bf16(BM, D, 1);
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool r = wait_bar_ctrl(b, parity, sh, p.err);
        return __all_sync(0xffffffffu, r ? 1 : 0) != 0;
    };
    // descriptors: Q of this slot (K-major), K/V stage 0 (K-major for S, MN-major for P V)
    const uint64_t dq = ptx::sdesc_sw128(sh.base + p.off_q[slot], 16, 1024);
    const uint64_t dk0 = ptx::sdesc_sw128(sh.base + p.off_kv, 16, 1024);
    const uint64_t dv0 = ptx::sdesc_sw128(sh.base + p.off_kv, BN * 128, 1024);
    const uint64_t stage16 = p.stage_bytes >> 4;
    const uint32_t tS = tmem + T::S(slot), tO = tmem + T::O(slot), tP = tmem + T::P(slot);
    const uint32_t tB = tmem + T::Bn(slot);
    // K-major operand, k-step kk of 16: 64-column block kk / 4 (rows x 128 bytes apart),
    // 32 bytes per step inside the 128-byte swizzle atom
    auto kstep = [](int kk, int rows) -> uint64_t {
        return (uint64_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
    };
    uint32_t kv_it = 0, q_it = 0, av_it = 0;
    uint32_t s_it = 0, p_it = 0, pv_it = 0, bn_it = 0, bd_it = 0;
    bool pv_pending = false;  // a P . V MMA (reading P over S) may still run
    bool bn_pending = false;  // a beta W^V MMA (reading the bins in the S columns) may still run
    bool ok = true;

    // before an MMA writes the slot's S columns: the softmax has read the previous S item,
    // and the MMAs reading P (P over S) or the value bins from those columns are done (MMAs
    // into different accumulators are not ordered among themselves). Each of the two waits
    // is for the latest commit on its barrier, so its parity is never two phases behind.
    auto claim_s = [&]() -> bool {
        if (bn_pending) {
            if (!wait(sbar(SB_BN_DONE), (bd_it - 1u) & 1u)) return false;
            bn_pending = false;
        }
        if (T::P_ALIAS && pv_pending) {
            if (!wait(sbar(SB_PV_DONE), (pv_it - 1u) & 1u)) return false;
            pv_pending = false;
        }
        if (!wait(sbar(SB_S_EMPTY), (s_it & 1u) ^ 1u)) return false;
        ++s_it;
        ptx::tc_fence_after();
        return true;
    };

    Sched sc(p, sh);
    for (int t = sc.next(p); t >= 0 && ok; t = sc.next(p)) {
        const Item it = decode_item(p, t);
        Plan<CAUSAL, EARLY_S> pl;
        pl.make(p, it);
        if (SPLIT) pl.keep_only(slot);
        if (pl.Jmax == 0) continue;
        const bool act = pl.active(slot);
        if (!(ok = wait(q_full, q_it & 1u))) break;
        ++q_it;
        ptx::tc_fence_after();
        int k_left = act ? pl.J[slot] : 0;  // S steps still to issue (Q is read until the last)
        if (!act) ptx::mbar_arrive_w(q_empty);
        if (AK && act) {  // R = Q W^K^T into the slot's S columns
            if (!(ok = claim_s())) break;
            const uint32_t idR = ptx::idesc_bf16(BM, (uint32_t)p.npad_k, 0);
            const uint64_t dak = ptx::sdesc_sw128(sh.base + p.off_ak[p.two_tables ? slot : 0], 16, 1024);
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::tc_mma_w(tS, dq + kstep(kk, BM), dak + kstep(kk, p.npad_k), idR, kk > 0 ? 1u : 0u);
            ptx::tc_commit_w(sbar(SB_S_FULL));
        }
        for (int g = 0; g < pl.groups() && ok; ++g) {
            for (int e = 0; e < 2 && ok; ++e) {
                bool isK;
                int j, mask, src;
                if (!pl.entry(g, e, isK, j, mask, src)) continue;
                uint32_t stg, round;
                ring_pos(p, kv_it, stg, round);
                stg += (uint32_t)ring0;
                ++kv_it;
                if (!(ok = wait(bar(B_KV0 + (int)stg), round & 1u))) break;
                const uint32_t empty = bar(B_KV0 + kMaxStages + (int)stg);
                if (!(mask & (1 << slot))) {  // the other slot's entry: release at once
                    ptx::mbar_arrive_w(empty);
                    continue;
                }
                ptx::tc_fence_after();
                const uint64_t off = (uint64_t)stg * stage16;
                const int cols = tile_cols(pl.nkc[slot], j);
                if (isK) {  // S_j = Q K_j^T
                    if (!(ok = claim_s())) break;
                    const uint32_t idS = ptx::idesc_bf16(BM, (uint32_t)cols, 0);
                    const uint64_t dk = dk0 + off;
                    // d = 128: one chain of 8 k-steps (one elect, immediate operand offsets);
                    // at d = 64 the rolled loop keeps the code small (its items are short)
                    if (D == 128) {
                        ptx::tc_mma_ss_k128(tS, dq, dk, idS, 0u);
                    } else {
#pragma unroll 1
                        for (int kk = 0; kk < D / 16; ++kk)
                            ptx::tc_mma_w(tS, dq + kstep(kk, BM), dk + kstep(kk, BN), idS, kk > 0 ? 1u : 0u);
                    }
                    ptx::tc_commit_w(sbar(SB_S_FULL));
                } else {  // O += P_j V_j
                    if (!(ok = wait(sbar(SB_P_FULL), p_it & 1u))) break;
                    ++p_it;
                    ptx::tc_fence_after();
                    const uint64_t dv = dv0 + off;
                    const int nk16 = cols / 16;
                    if (D == 128 && nk16 == BN / 16) {  // a whole tile: one chain of 8 k-steps
                        ptx::tc_mma_ts_k128(tO, tP, dv, idPV, j > 0 ? 1u : 0u);
                    } else {
#pragma unroll 1
                        for (int kk = 0; kk < nk16; ++kk)
                            ptx::tc_mma_ts_w(tO, tP + (uint32_t)(kk * 8), dv + (uint64_t)(kk * 16 * 128 >> 4),
                                             idPV, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit_w(sbar(SB_PV_DONE));
                    ++pv_it;
                    pv_pending = true;
                }
                ptx::tc_commit_w(empty);  // the entry is free once these MMAs are done
                if (isK && --k_left == 0) ptx::tc_commit_w(q_empty);  // last read of Q
            }
        }
        if (!ok) break;
        if (AV) {  // O += beta W^V, beta (bf16 pairs) in the upper S columns of the slot
            if (!(ok = wait(av_full, av_it & 1u))) break;
            ++av_it;
            if (act) {
                if (!(ok = wait(sbar(SB_BN_FULL), bn_it & 1u))) break;
                ++bn_it;
                ptx::tc_fence_after();
                const uint64_t dav = ptx::sdesc_sw128(sh.base + p.off_av[p.two_tables ? slot : 0],
                                                      (uint32_t)p.kpad_v * 128, 1024);
#pragma unroll 1
                for (int kk = 0; kk < p.kpad_v / 16; ++kk)
                    ptx::tc_mma_ts_w(tO, tB + (uint32_t)(kk * 8), dav + (uint64_t)(kk * 16 * 128 >> 4), idPV, 1u);
                ptx::tc_commit_w(sbar(SB_BN_DONE));
                ++bd_it;
                bn_pending = true;
                ptx::tc_commit_w(av_empty);
            } else {
                ptx::mbar_arrive_w(av_empty);
            }
        }
        if (act) ptx::tc_commit_w(sbar(SB_O_FULL));
    }
    // every MMA issued by this warp completes before TMEM is released
    ptx::tc_commit_w(sbar(SB_DRAIN));
    drain_bar(sbar(SB_DRAIN), 0, sh.limit);
}

// ======================================================================= softmax / epilogue
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return ptx::pack_bf16x2(lo, hi); }

// Element pairs (e, e + 1) of a register array go through the two-lane fp32 instructions
// (one issue for two fused multiply-adds, adds or multiplies, each rounded as its scalar form)
__device__ __forceinline__ float2 pair(const float *x, int e) { return make_float2(x[e], x[e + 1]); }
__device__ __forceinline__ void put(float *x, int e, float2 v) {
    x[e] = v.x;
    x[e + 1] = v.y;
}
__device__ __forceinline__ float2 dup(float v) { return make_float2(v, v); }

// maximum of 32 values, 16 three-input instructions, depth 5
__device__ __forceinline__ float max32(const float *x) {
    float a0 = ptx::max3(x[0], x[1], x[2]), a1 = ptx::max3(x[3], x[4], x[5]);
    float a2 = ptx::max3(x[6], x[7], x[8]), a3 = ptx::max3(x[9], x[10], x[11]);
    a0 = ptx::max3(a0, x[12], x[13]);
    a1 = ptx::max3(a1, x[14], x[15]);
    a2 = ptx::max3(a2, x[16], x[17]);
    a3 = ptx::max3(a3, x[18], x[19]);
    a0 = ptx::max3(a0, x[20], x[21]);
    a1 = ptx::max3(a1, x[22], x[23]);
    a2 = ptx::max3(a2, x[24], x[25]);
    a3 = ptx::max3(a3, x[26], x[27]);
    a0 = ptx::max3(a0, x[28], x[29]);
    a1 = ptx::max3(a1, x[30], x[31]);
    return ptx::max3(a0, a1, fmaxf(a2, a3));
}
template <int D, bool SG, bool AK, bool AV, bool T5, bool CAUSAL>
__device__ void softmax_role(const Params &p, const Shared &sh, uint32_t tmem, int slot_in) {
    using T = Tm<D, SG>;
    const int slot = __shfl_sync(0xffffffffu, slot_in, 0);  // known warp-uniform from here on
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // warp-level values go through a full-warp broadcast: the compiler then knows them (and
    // every branch on them) to be warp-uniform, which keeps the per-chunk control flow free of
    // divergence handling
    auto uni = [](int v) { return __shfl_sync(0xffffffffu, v, 0); };
    const int quad = uni(warp & 3);  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const int stid = threadIdx.x - 32 * (kSoftWarp0 + 4 * slot);  // 0 .. 127
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t bars = sh.base + p.off_bar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    auto sbar = [&](int which) { return bar(B_SLOT0 + kSlotBars * slot + which); };
    float *Rrow = reinterpret_cast<float *>(sh.ptr + p.off_r[slot]) + row * p.SR;
    float *brow = reinterpret_cast<float *>(sh.ptr + p.off_beta[slot]) + row * p.SB;
    // T5 offset table, indices -kT5Pad .. 2R + kT5Pad (the ends repeat the saturated buckets,
    // so the banded gather of a chunk never clamps)
    float *t5tab = reinterpret_cast<float *>(sh.ptr + p.off_t5[slot]) + kT5Pad;
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.f;  // raw chunks need max(x * sl2) = sl2 * max(x)
    const int k = p.clip_k;
    const int hi_off = CAUSAL ? 0 : k;  // largest offset held in the staged table rows
    const int W = p.W;
    uint32_t s_it = 0, pv_it = 0, o_it = 0;
    int t5_head = -1;
    bool ok = true;
    // tcgen05.ld/st are warp-collective (.sync.aligned): every decision guarding them is
    // uniform across the warp, and the warp reconverges before each TMEM access.
    // Only the slot's first warp polls the mbarrier; the other three wait for it at the
    // slot's named barrier, which carries the outcome to all 128 threads.
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        bool r = true;
        if (quad == 0) {
            r = wait_bar(b, parity, sh, p.err);
            r = __all_sync(0xffffffffu, r ? 1 : 0) != 0;
        }
        return slot_sync(slot, r);
    };
    auto wait_s = [&]() -> bool {
        if (!wait_w(sbar(SB_S_FULL), s_it & 1u)) return false;
        ++s_it;
        ptx::tc_fence_after();
        __syncwarp();
        return true;
    };
    auto release_s = [&]() {
        ptx::tc_fence_before();
        ptx::mbar_arrive(sbar(SB_S_EMPTY));
    };
    // completion number c of the slot's P-reading MMAs (waited in increasing order; the
    // next completion needs a P item this thread has not written yet)
    auto wait_pv = [&](uint32_t c) -> bool {
        if (!wait_w(sbar(SB_PV_DONE), c & 1u)) return false;
        ptx::tc_fence_after();
        __syncwarp();
        return true;
    };
    auto rel = [&](int idx) -> float { return Rrow[idx]; };  // scaled R value of table row idx

    // the next item is decoded and its key count loaded while the current one runs
    Sched sc(p, sh);
    int t_next = sc.next(p);
    SlotItem nxt = slot_item(p, t_next, slot);
    for (int t = t_next; t >= 0 && ok; t = t_next) {
        const SlotItem cur = nxt;
        t_next = sc.next(p);
        nxt = slot_item(p, t_next, slot);
        if (!cur.valid) continue;
        const int bh = uni(cur.bh), qt = uni(cur.qt);
        const int i0 = qt * BM, gi = i0 + row, h = bh % p.H;
        const int gmin = uni(i0 + quad * 32), gmax = gmin + 31;  // rows of this warp
        const int nk = uni(cur.nk);
        const int nkc = CAUSAL ? min(nk, i0 + BM) : nk;  // keys any row of the tile may see
        const int J = (nkc + BN - 1) / BN;
        __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                              ((long long)bh * p.n + gi) * D;
        if (J == 0) {
            if (gi < p.n) {
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                    reinterpret_cast<uint4 *>(orow)[c] = make_uint4(0, 0, 0, 0);
            }
            continue;
        }
        if (T5 && h != t5_head) {
            if (!(ok = slot_sync(slot, true))) break;  // every row is done with the old table
            for (int idx = stid - kT5Pad; idx <= 2 * p.t5_R + kT5Pad; idx += 128)
                t5tab[idx] = scalar_bias(p.bias, p.bias_kind, p.H, p.bias_R, p.bias_hs, p.t5,
                                         idx - p.t5_R, h) * kLog2e;
            if (!(ok = slot_sync(slot, true))) break;
            t5_head = h;
        }
        if (AK) {  // R row -> shared memory (scaled to the log2 domain)
            if (!(ok = wait_s())) break;
            for (int c0 = 0; c0 < p.npad_k; c0 += 16) {
                uint32_t r[16];
                ptx::tmem_ld16(lane_base + T::S(slot) + (uint32_t)c0, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c0 + e < W) Rrow[c0 + e] = __uint_as_float(r[e]) * sl2;
            }
            release_s();
        }
        // relative term of keys beyond the window on either side (constant per row)
        float c_left = 0.f, c_right = 0.f;
        if (AK) {
            c_left = rel(0);
            c_right = rel(W - 1);
        } else if (T5) {
            c_left = t5tab[0];
            c_right = t5tab[2 * p.t5_R];
        }
        // offsets at or beyond these take the first / last table row
        const int lo_lim = T5 ? -p.t5_R : -k;
        const int hi_lim = T5 ? p.t5_R : hi_off;
        if (AV)
            for (int r = 0; r < W; ++r) brow[r] = 0.f;
        float m_ref = -INFINITY, l = 0.f, lsum = 0.f;

        for (int j = 0; j < J; ++j) {
            const int j0 = j * BN;
            const int cols = tile_cols(nkc, j);  // multiple of 32, > 0
            int live = cols / KB;                 // chunks any row of the warp can see
            if (CAUSAL) live = min(live, max(0, (gmax - j0) / KB + 1));
            if (!(ok = wait_s())) break;
            // ---- the score row into registers, then the buffer goes back to the MMA warp
            float x[BN];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                if (c < live) ptx::tmem_ld32f(lane_base + T::S(slot) + (uint32_t)(c * KB), x + c * KB);
            ptx::tmem_ld_wait();
            // with value bins, the last tile's S columns are kept for them (released below)
            if (!AV || j + 1 < J) release_s();
            // ---- logits in the log2 domain (S2-S4). A chunk whose relative term is one
            // constant for every row of the warp and that needs no mask stays raw (for a
            // non-negative scale): its exponent is x * sl2 + (c - m), and its maximum comes
            // from the raw maximum. Other chunks get the full logit (gathered relative term,
            // masks) written in place and exponent x - m.
            // chunk c of the tile: is it kept raw, and with which constant
            auto raw_chunk = [&](int c, float &cst) -> bool {
                const int e0 = j0 + c * KB;  // first key of the chunk
                // offsets j - i over the warp's rows lie in [e0 - gmax, e0 + 31 - gmin]
                const bool w_left = (e0 + KB - 1 - gmin) <= lo_lim;
                const bool w_right = (e0 - gmax) >= hi_lim;
                const bool uniform = (!AK && !T5) || w_left || w_right;
                const bool full = (e0 + KB <= nk) && (!CAUSAL || e0 + KB - 1 <= gmin);
                cst = (!AK && !T5) ? 0.f : (w_left ? c_left : c_right);
                return uniform && full && pos_scale;
            };
            float rmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if (c >= live) continue;
                float *xc = x + c * KB;
                float cst;
                if (raw_chunk(c, cst)) {
                    rmax = fmaxf(rmax, fmaf(max32(xc), sl2, cst));
                    continue;
                }
                const int e0 = j0 + c * KB;
                const bool w_left = (e0 + KB - 1 - gmin) <= lo_lim;
                const bool w_right = (e0 - gmax) >= hi_lim;
                const bool full = (e0 + KB <= nk) && (!CAUSAL || e0 + KB - 1 <= gmin);
                const int base = e0 - gi;  // offset of element 0 for this row
                if (AK) {
                    if (w_left || w_right) {
                        const float2 cst = dup(w_left ? c_left : c_right);
#pragma unroll
                        for (int e = 0; e < KB; e += 2) put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), cst));
                    } else {
                        const int rb = base + k;  // table row of element 0, before clamping
#pragma unroll
                        for (int e = 0; e < KB; e += 2) {
                            const float2 r = make_float2(rel(min(W - 1, max(0, rb + e))),
                                                         rel(min(W - 1, max(0, rb + e + 1))));
                            put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), r));
                        }
                    }
                } else if (T5) {
                    const int R = p.t5_R;
                    if (w_left || w_right) {
                        const float2 cst = dup(w_left ? c_left : c_right);
#pragma unroll
                        for (int e = 0; e < KB; e += 2) put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), cst));
                    } else {
                        const int tb = base + R;
#pragma unroll
                        for (int e = 0; e < KB; e += 2) {
                            const float2 r = make_float2(t5tab[tb + e], t5tab[tb + e + 1]);
                            put(xc, e, __ffma2_rn(pair(xc, e), dup(sl2), r));
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < KB; e += 2) put(xc, e, __fmul2_rn(pair(xc, e), dup(sl2)));
                }
                if (!full) {  // keys j < nk (and j <= i when causal): e < lim
                    const int lim = (CAUSAL ? min(nk, gi + 1) : nk) - e0;
#pragma unroll
                    for (int e = 0; e < KB; ++e) xc[e] = e < lim ? xc[e] : -INFINITY;
                }
                rmax = fmaxf(rmax, max32(xc));
            }
            // ---- online softmax (S5) with a lazy rescale
            float alpha = 1.f;
            if (rmax > m_ref + kRescaleLog2) {
                alpha = ptx::ex2(m_ref - rmax);  // 0 while nothing was seen yet
                m_ref = rmax;
            }
            // P and O of the slot are free once the previous P . V is done (with P over S that
            // is already so: S_j was issued only after that P . V had completed)
            if (!T::P_ALIAS && j >= 1 && !(ok = wait_pv(pv_it + (uint32_t)j - 1u))) break;
            // on the first key tile l, the bins and O hold nothing yet: no rescale needed
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                l *= alpha;
                lsum *= alpha;
                if (AV && alpha != 1.f)
                    for (int r = 0; r < W; ++r) brow[r] *= alpha;
                __syncwarp();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t r[32];
                    ptx::tmem_ld32(lane_base + T::O(slot) + (uint32_t)c0, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 v = __fmul2_rn(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                                    dup(alpha));
                        r[e] = __float_as_uint(v.x);
                        r[e + 1] = __float_as_uint(v.y);
                    }
                    ptx::tmem_st32(lane_base + T::O(slot) + (uint32_t)c0, r);
                }
                ptx::tmem_st_wait();
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            // ---- exponentials, row sum, value bins (S7), P (bf16 pairs) into TMEM
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if (c * KB >= cols) continue;  // never read by P V
                // P (bf16 pairs) is packed into the chunk's own score registers, which are dead
                // by then, so the asynchronous TMEM store of one chunk never holds registers
                // that the next chunk writes
                float *xc = x + c * KB;
                if (c >= live) {  // no row of this warp sees these keys
#pragma unroll
                    for (int e = 0; e < KB / 2; ++e) xc[e] = 0.f;
                } else {
                    float cst;
                    const bool rawc = raw_chunk(c, cst);
                    const float a = rawc ? sl2 : 1.f, b = (rawc ? cst : 0.f) - m_use;
                    const float2 a2 = dup(a), b2 = dup(b);
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
                        // bins 1 .. W-1 get exactly one key each over the whole row (offsets
                        // -k+1 .. hi_off) and are stored as they come. The end bins come from
                        // sums at the end of the row: bin 0 from l (causal) or from lsum, the
                        // keys at or left of the diagonal (not causal), which also gives bin W-1
                        const int e0 = j0 + c * KB;
                        if (!CAUSAL) {
                            if (e0 + KB <= gmin) {  // left of every row's diagonal
                                lsum += rs;
                            } else if (e0 == gmin) {  // the warp's diagonal chunk: keys j <= i
#pragma unroll
                                for (int e = 0; e < KB; ++e) lsum += e <= lane ? xc[e] : 0.f;
                            }
                        }
                        // chunks whose keys all fall in an end bin for every row need nothing
                        const bool w_left = (e0 + KB - 1 - gmin) <= -k;
                        const bool w_right = CAUSAL ? e0 > gmax : (e0 - gmax) >= k;
                        if (!w_left && !w_right) {
                            float *bp = brow + (e0 - gi + k);  // bin of element 0
                            const int elo = gi - k - e0;  // elements elo .. elo + W - 1: bins 0 .. W-1
#pragma unroll
                            for (int e = 0; e < KB; ++e)
                                if ((unsigned)(e - elo) < (unsigned)W) bp[e] = xc[e];
                        }
                    }
#pragma unroll
                    for (int e = 0; e < KB / 2; ++e)
                        xc[e] = __uint_as_float(pack2(xc[2 * e], xc[2 * e + 1]));
                }
                __syncwarp();
                ptx::tmem_st16f(lane_base + T::P(slot) + (uint32_t)(c * (KB / 2)), xc);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(sbar(SB_P_FULL));
        }
        if (!ok) break;
        pv_it += (uint32_t)J;  // P . V completions of this item
        if (AV) {
            // bins (bf16 pairs) become the A operand of O += beta W^V; that MMA is issued after
            // the last P . V by the same thread and runs after it
            if (!CAUSAL && W > 1) {
                // lsum = bin 0 + bins 1 .. k; l - lsum = bins k+1 .. W-2 + bin W-1
                float a = 0.f, b = 0.f;
                for (int r = 1; r <= k; ++r) a += brow[r];
                for (int r = k + 1; r < W - 1; ++r) b += brow[r];
                brow[0] = fmaxf(0.f, lsum - a);
                brow[W - 1] = fmaxf(0.f, (l - lsum) - b);
            } else {  // l = bin 0 + bins 1 .. W-1
                float a = 0.f, b = 0.f;
                int r = 1;
                for (; r + 1 < W; r += 2) {
                    a += brow[r];
                    b += brow[r + 1];
                }
                if (r < W) a += brow[r];
                brow[0] = fmaxf(0.f, l - (a + b));
            }
            for (int c0 = 0; c0 < p.kpad_v; c0 += 32) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r0 = c0 + 2 * e;
                    pk[e] = pack2(r0 < W ? brow[r0] : 0.f, r0 + 1 < W ? brow[r0 + 1] : 0.f);
                }
                __syncwarp();
                ptx::tmem_st16(lane_base + T::Bn(slot) + (uint32_t)(c0 / 2), pk);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            // a barrier of their own: nothing orders this arrival after the MMA warp has seen
            // the last P tile, so on P_FULL it could complete the next phase before that
            ptx::mbar_arrive(sbar(SB_BN_FULL));
            ptx::mbar_arrive(sbar(SB_S_EMPTY));  // the S columns go back once the bins are read
        }
        // ---- epilogue (S8): O / l -> bf16 -> global
        if (!(ok = wait_w(sbar(SB_O_FULL), o_it & 1u))) break;
        ++o_it;
        ptx::tc_fence_after();
        __syncwarp();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        // the O row in halves of 64 columns (one TMEM wait per half)
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t r[64];
            ptx::tmem_ld32(lane_base + T::O(slot) + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[32]>(r));
            ptx::tmem_ld32(lane_base + T::O(slot) + (uint32_t)c0 + 32u,
                           *reinterpret_cast<uint32_t(*)[32]>(r + 32));
            ptx::tmem_ld_wait();
            if (gi < p.n) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 o = __fmul2_rn(make_float2(__uint_as_float(r[8 * q + 2 * h]),
                                                                __uint_as_float(r[8 * q + 2 * h + 1])),
                                                    dup(inv));
                        w[h] = pack2(o.x, o.y);
                    }
                    reinterpret_cast<uint4 *>(orow)[c0 / 8 + q] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            __syncwarp();
        }
        ptx::tc_fence_before();
    }
}

// ======================================================================= kernel
template <int D, bool SG, bool AK, bool AV, bool T5, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    relattn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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
    const uint32_t bars = sh.base + p.off_bar;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i >= B_SLOT0 && i < B_KV0) {
                const int which = (i - B_SLOT0) % kSlotBars;
                if (which == SB_S_EMPTY || which == SB_P_FULL || which == SB_BN_FULL)
                    cnt = 128;  // the slot's threads
            }
            // shared feed: released by both MMA warps
            if (i == B_Q_EMPTY || i == B_AV_EMPTY || (!p.split && i >= B_KV0 + kMaxStages)) cnt = 2;
            ptx::mbar_init(bars + 8u * (uint32_t)i, cnt);
        }
        *sh.abort_flag = 0;
        if (p.snake) snake_list(p, reinterpret_cast<int *>(sh.ptr + p.off_list));
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
    // warp is converged and the value warp-uniform, so tcgen05 and TMA operands stay in uniform
    // registers and each such instruction is a single issue.
    if (warp < kSoftWarp0) {
        ptx::reg_dealloc<kCtrlRegs>();
        if (warp == 0 || (p.split && warp == 3)) {  // split feed: warp 3 feeds slot 1
            (void)__shfl_sync(0xffffffffu, tmem_raw, 0);
            producer_role<D, SG, AK, AV, CAUSAL>(p, sh, &tm_q, &tm_k, &tm_v, &tm_kf, &tm_vf, &tm_ak,
                                             &tm_av, warp == 3 ? 1 : 0);  // the whole warp; one lane issues
        } else if (warp == 1 || warp == 2) {
            const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_raw, 0);
            mma_role<D, SG, AK, AV, CAUSAL>(p, sh, tmem, warp - 1);  // slot warp - 1; one lane issues
        }
        __syncwarp();
    } else {
        ptx::reg_alloc<kSoftRegs>();
        const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_raw, 0);
        softmax_role<D, SG, AK, AV, T5, CAUSAL>(p, sh, tmem, (warp - kSoftWarp0) >> 2);
    }

    ptx::tc_fence_before();
    ptx::cta_barrier();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_raw, 512);
    }
}

}  // namespace tc
}  // namespace relattn
