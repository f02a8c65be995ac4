// Host side of the tcgen05 path: shared-memory layout, TMA descriptors, variant
// selection and launch. Included by relattn_tc_d64.cu / relattn_tc_d128.cu, which each
// instantiate one head dimension.
#pragma once

#include <cstdio>
#include <cstring>
#include <mutex>

#include "relattn_tc_kernel.cuh"

namespace relattn {
namespace tc {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 3-D bf16 map over [dim2][dim1][dim0] (dim0 contiguous), box {64, box1, 1}, 128-byte
// swizzle, out-of-range elements read as zero (and are not written by stores).
inline bool make_map(CUtensorMap *m, const void *ptr, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                     uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t gdim[3] = {dim0, dim1, dim2};
    const cuuint64_t gstride[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {64, box1, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), gdim, gstride, box,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;      // max dynamic shared memory of one block
    int smem_per_sm = 0;     // shared memory of one SM
    int smem_reserved = 0;   // shared memory the system keeps per block
    int l2_bytes = 0;
};

inline DeviceInfo device_info() {
    static DeviceInfo cache[64];
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return DeviceInfo{};
    if (cache[dev].sms == 0) {
        cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&cache[dev].smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&cache[dev].smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&cache[dev].smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        cudaDeviceGetAttribute(&cache[dev].l2_bytes, cudaDevAttrL2CacheSize, dev);
    }
    return cache[dev];
}

inline uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int D, bool SG, bool AK, bool AV, bool T5, bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap (&tm)[7], const Params &p, uint32_t smem_bytes,
                           cudaStream_t s) {
    auto kern = relattn_tc_kernel<D, SG, AK, AV, T5, CAUSAL>;
    // Opt in to the device's whole shared-memory budget once per device and variant, so
    // that later calls (including ones captured into a CUDA graph) only launch.
    static bool opted[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const DeviceInfo di = device_info();
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opted[dev]) {
            // the warpgroups' register shares add up to kThreads * kLaunchRegs: launching
            // with fewer registers per thread would leave the softmax warps waiting for
            // registers that never come
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kern);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != kLaunchRegs) return cudaErrorNotSupported;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
            opted[dev] = true;
        }
    }
    const int grid = p.num_items < di.sms ? p.num_items : di.sms;  // persistent: one CTA per SM
    kern<<<grid, kThreads, smem_bytes, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], tm[6], p);
    return cudaGetLastError();
}

template <int D, bool SG, bool T5, bool CAUSAL>
cudaError_t launch_terms(bool ak, bool av, const CUtensorMap (&tm)[7], const Params &p,
                         uint32_t smem, cudaStream_t s) {
    if constexpr (T5) {
        return launch_variant<D, SG, false, false, true, CAUSAL>(tm, p, smem, s);
    } else {
        if (ak && av) return launch_variant<D, SG, true, true, false, CAUSAL>(tm, p, smem, s);
        if (ak) return launch_variant<D, SG, true, false, false, CAUSAL>(tm, p, smem, s);
        if (av) return launch_variant<D, SG, false, true, false, CAUSAL>(tm, p, smem, s);
        return launch_variant<D, SG, false, false, false, CAUSAL>(tm, p, smem, s);
    }
}

// Shared-memory layout for `stages` K/V stages (p.pair, p.two_tables and p.SR set);
// returns the bytes to request.
template <int D>
inline uint32_t layout(Params &p, bool ak, bool av, bool t5mode, int stages) {
    const int nslots = p.pair ? 2 : 1;
    const int ntab = p.two_tables ? 2 : 1;
    const uint32_t q_bytes = (uint32_t)BM * D * 2;
    const uint32_t stage_bytes = (uint32_t)BN * D * 2;
    const uint32_t r_bytes = round_up((uint32_t)BM * p.SR * 4, 16);
    const uint32_t b_bytes = round_up((uint32_t)BM * p.SB * 4, 16);
    const uint32_t t_bytes = round_up((uint32_t)(2 * p.t5_R + 1 + 2 * kT5Pad) * 4, 16);
    uint32_t off = 0;
    // TMA targets first: every size below is a multiple of 1024 bytes
    for (int s = 0; s < 2; ++s) {
        p.off_q[s] = off;
        if (s < nslots) off += q_bytes;
    }
    p.off_kv = off;
    off += (uint32_t)stages * stage_bytes;
    for (int s = 0; s < 2; ++s) {
        p.off_ak[s] = s < ntab ? off : p.off_ak[0];
        if (ak && s < ntab) off += (uint32_t)p.npad_k * D * 2;
    }
    for (int s = 0; s < 2; ++s) {
        p.off_av[s] = s < ntab ? off : p.off_av[0];
        if (av && s < ntab) off += (uint32_t)p.kpad_v * D * 2;
    }
    for (int s = 0; s < 2; ++s) {
        p.off_r[s] = off;
        if (ak && s < nslots) off += r_bytes;
    }
    for (int s = 0; s < 2; ++s) {
        p.off_beta[s] = off;
        if (av && s < nslots) off += b_bytes;
    }
    for (int s = 0; s < 2; ++s) {
        p.off_t5[s] = off;
        if (t5mode && s < nslots) off += t_bytes;
    }
    p.off_bar = off;
    off += (uint32_t)kNumBars * 8 + 16;
    p.off_list = off;  // the snake-order item list (used only when p.snake)
    off += (uint32_t)kListCap * 4;
    p.stages = stages;
    // split feed with two slots: each slot's ring takes half of the stages
    const int rs = p.split ? stages / 2 : stages;
    p.ring_stages = rs;
    p.stage_bytes = stage_bytes;
    p.stage_mul = rs > 0 ? (uint32_t)((0x100000000ull + (uint64_t)rs - 1) / (uint64_t)rs) : 0u;
    return off + 1024;  // slack to align the base to 1024 bytes
}

template <int D>
cudaError_t launch_tc(const TcArgs &a, const T5Buckets *t5, int *err_word, cudaStream_t s) {
    const bool t5mode = a.mode == kT5;
    const bool ak = !t5mode && a.aK != nullptr;
    const bool av = !t5mode && a.aV != nullptr;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.BH = a.B * a.H;
    p.H = a.H;
    p.n = a.n;
    p.n_qtiles = (a.n + BM - 1) / BM;
    p.scale_log2 = a.scale * kLog2e;
    p.kv_len = a.kv_len;
    p.err = err_word;
    p.out = a.out;
    p.clip_k = a.clip_k;
    p.W = 1;
    if (ak || av) {
        p.W = a.causal ? a.clip_k + 1 : 2 * a.clip_k + 1;
        if (p.W > 128) return cudaErrorNotSupported;
    }
    p.SB = (p.W + 2) & ~1;  // even, > W: conflict-free bin gathers and a spare slot
    p.npad_k = (int)round_up((uint32_t)p.W, 16);
    p.kpad_v = p.npad_k;
    p.table_heads = a.ths != 0 ? 1 : 0;
    p.bias = a.bias;
    if (t5mode) {
        // the shared-memory table covers offsets -t5_R .. t5_R; beyond them the bias is
        // constant (T5: the saturated buckets; a clipped table: its end entries). ALiBi never
        // saturates: its table spans every offset of the sequence.
        p.bias_kind = a.bias_kind;
        p.bias_R = a.bias_R;
        p.bias_hs = a.bias_hs;
        if (a.bias_kind == kBiasBuckets) {
            if (!t5) return cudaErrorInvalidValue;
            p.t5 = *t5;
            p.t5_R = t5->sat;
        } else if (a.bias_kind == kBiasAlibi) {
            p.t5_R = a.n - 1;
        } else {
            p.t5_R = a.bias_R < a.n - 1 ? a.bias_R : a.n - 1;
        }
    }
    // no shared-memory table over 2^17 offsets fits (and 2 * t5_R stays in range)
    if (t5mode && (p.t5_R < 0 || p.t5_R > (1 << 16))) return cudaErrorNotSupported;
    if (p.BH == 0 || p.n_qtiles == 0) return cudaSuccess;

    const DeviceInfo di = device_info();
    if (di.sms <= 0 || di.smem_optin <= 0) return cudaErrorInvalidDevice;
    // schedule heads in groups whose K and V fit in half of L2
    {
        const int64_t per_head = 2LL * a.n * D * 2;
        const int64_t fit = di.l2_bytes > 0 ? (int64_t)di.l2_bytes / 2 / (per_head > 0 ? per_head : 1) : p.BH;
        p.head_group = (int)(fit < 1 ? 1 : (fit > p.BH ? p.BH : fit));
    }
    // Choose the first configuration that fits shared memory: two query tiles per item
    // before one, three K/V stages before two. Heads of one query tile pair two heads per
    // item with nothing to share between the slots: they take the split feed first (two
    // stages per slot).
    struct Choice { int pair, split, min_stages; };
#ifndef RELATTN_D128_PAIR_FIRST
#define RELATTN_D128_PAIR_FIRST 1
#endif
    const Choice pair_first[] = {{1, 1, 4}, {1, 0, 3}, {1, 0, 2}, {0, 0, 3}, {0, 0, 2}};
    const Choice single_first[] = {{0, 0, 3}, {0, 0, 2}, {1, 0, 3}, {1, 0, 2}, {1, 0, 2}};
    const Choice *choices = (D == 128 && !RELATTN_D128_PAIR_FIRST) ? single_first : pair_first;
    // R rows (fp32): an even stride, so that W - 1 + stride is odd and the banded gathers of
    // the 32 rows of a warp fall in 32 distinct banks
    p.SR = p.W + (p.W & 1);
    uint32_t smem = 0;
    bool found = false;
    for (int ci = 0; ci < 5; ++ci) {
        const Choice &c = choices[ci];
        if (c.split && p.n_qtiles != 1) continue;
        Params q = p;
        q.pair = c.pair;
        q.split = c.split;
        // the two tiles of an item belong to different heads only for odd tile counts; with
        // the split feed each slot loads its own tables anyway
        q.two_tables = (c.pair && (ak || av) &&
                        (c.split || ((p.n_qtiles & 1) && p.table_heads))) ? 1 : 0;
        const uint32_t fixed = layout<D>(q, ak, av, t5mode, 0);
        int64_t st = ((int64_t)di.smem_optin - (int64_t)fixed) / ((int64_t)BN * D * 2);
        if (st > kMaxStages) st = kMaxStages;
        if (c.split) st &= ~(int64_t)1;  // two rings of equal size
        if (st < c.min_stages) continue;
        p = q;
        smem = layout<D>(p, ak, av, t5mode, (int)st);
        found = true;
        break;
    }
    if (!found || smem > (uint32_t)di.smem_optin) return cudaErrorNotSupported;
    p.wait_limit = a.wait_limit > 0 ? a.wait_limit : 2000000000ll;
    p.withhold_q = a.withhold_q;
    {
        const int G = p.head_group;
        const int full = p.BH / G, rest = p.BH - full * G;
        const int64_t items = (int64_t)full * items_per_group(G, p.n_qtiles, p.pair) +
                              (rest ? items_per_group(rest, p.n_qtiles, p.pair) : 0);
        if (items > INT32_MAX) return cudaErrorNotSupported;
        p.num_items = (int)items;
        p.items_full = items_per_group(G, p.n_qtiles, p.pair);
        p.n_groups = full + (rest ? 1 : 0);
        const int grid = p.num_items < di.sms ? p.num_items : di.sms;  // as launched below
        p.rot_step = grid > 0 ? p.items_full % grid : 0;
        if ((int64_t)p.n_groups * grid > INT32_MAX) return cudaErrorNotSupported;  // g * rot_step
        // causal query tiles of one head differ in length when a head has more than one pair;
        // the order goes through a list of kListCap entries per CTA
        const int64_t per_cta = grid > 0 ? ((int64_t)p.num_items + grid - 1) / grid + p.n_groups : 0;
        p.snake = (a.causal && a.kv_len == nullptr && p.n_qtiles > 2 && per_cta + 1 < kListCap) ? 1 : 0;
        // a last wave of two-tile items that fills at most half of the grid runs as one-tile
        // items on twice as many CTAs (bidirectional only: a causal pair's tiles differ in
        // length and measured slower split)
        p.tail_from = p.num_items;
        if (p.pair && !a.causal && p.num_items >= di.sms) {
            const int r = p.num_items % di.sms;
            if (r > 0 && 2 * r <= di.sms) {
                p.tail_from = p.num_items - r;
                p.num_items = p.tail_from + 2 * r;
            }
        }
    }

    // ---- TMA descriptors (the output is written with plain stores)
    // q; k and v in 32-row boxes; k and v in whole-tile boxes; the two edge tables
    CUtensorMap tm[7];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    if (!make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !make_map(&tm[1], a.k, d, n, BH, rs, hs, KB) ||
        !make_map(&tm[2], a.v, d, n, BH, rs, hs, KB) || !make_map(&tm[3], a.k, d, n, BH, rs, hs, BN) ||
        !make_map(&tm[4], a.v, d, n, BH, rs, hs, BN))
        return cudaErrorInvalidValue;
    tm[5] = tm[0];
    tm[6] = tm[0];
    const uint64_t rows = (uint64_t)(2 * a.clip_k + 1);
    const uint64_t Ht = p.table_heads ? (uint64_t)a.H : 1;
    const uint64_t ths_bytes = p.table_heads ? (uint64_t)a.ths * 2 : rows * d * 2;
    if (ak && !make_map(&tm[5], a.aK, d, rows, Ht, rs, ths_bytes, (uint32_t)p.npad_k))
        return cudaErrorInvalidValue;
    if (av && !make_map(&tm[6], a.aV, d, rows, Ht, rs, ths_bytes, (uint32_t)p.kpad_v))
        return cudaErrorInvalidValue;

    // d = 128 with one tile per item keeps P in its own TMEM columns (layout SG)
    if (D == 128 && !p.pair) {
        if (a.causal)
            return t5mode ? launch_terms<D, true, true, true>(ak, av, tm, p, smem, s)
                          : launch_terms<D, true, false, true>(ak, av, tm, p, smem, s);
        return t5mode ? launch_terms<D, true, true, false>(ak, av, tm, p, smem, s)
                      : launch_terms<D, true, false, false>(ak, av, tm, p, smem, s);
    }
    if (a.causal)
        return t5mode ? launch_terms<D, false, true, true>(ak, av, tm, p, smem, s)
                      : launch_terms<D, false, false, true>(ak, av, tm, p, smem, s);
    return t5mode ? launch_terms<D, false, true, false>(ak, av, tm, p, smem, s)
                  : launch_terms<D, false, false, false>(ak, av, tm, p, smem, s);
}

}  // namespace tc
}  // namespace relattn
