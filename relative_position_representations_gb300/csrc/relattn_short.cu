// Host side of the short-sequence kernel (relattn_short.cuh): shared-memory layout, ring
// sizes, TMA descriptors, variant selection and launch. Sequences of at most 256 keys, head
// dimension 64, bf16, the Shaw edge tables (either, both or none) with at most 64 staged
// rows; the caller takes the long-sequence kernel for anything else.
#include "relattn_short.cuh"
#include "relattn_tc_launch.cuh"

namespace relattn {
namespace sk {

template <bool AK, bool AV, bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap (&tm)[8], const Params &p, uint32_t smem_bytes, int grid,
                           cudaStream_t s) {
    auto kern = relattn_short_kernel<AK, AV, CAUSAL>;
    // opt in to the shared memory once per device and variant, so that later calls (including
    // ones captured into a CUDA graph) only launch
    static bool opted[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opted[dev]) {
            // the groups' register shares add up to kThreads * kLaunchRegs: launching with fewer
            // registers per thread would leave the softmax warps waiting for registers
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kern);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != kLaunchRegs) return cudaErrorNotSupported;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     tc::device_info().smem_optin);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
            opted[dev] = true;
        }
    }
    kern<<<grid, kThreads, smem_bytes, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], tm[6], tm[7], p);
    return cudaGetLastError();
}

template <bool CAUSAL>
cudaError_t launch_terms(bool ak, bool av, const CUtensorMap (&tm)[8], const Params &p, uint32_t smem,
                         int grid, cudaStream_t s) {
    if (ak && av) return launch_variant<true, true, CAUSAL>(tm, p, smem, grid, s);
    if (ak) return launch_variant<true, false, CAUSAL>(tm, p, smem, grid, s);
    if (av) return launch_variant<false, true, CAUSAL>(tm, p, smem, grid, s);
    return launch_variant<false, false, CAUSAL>(tm, p, smem, grid, s);
}

// Shared memory for ks K stages and vs V stages; returns the bytes to request. TMA targets
// first (every size a multiple of 1024 bytes): Q, the K and V rings, W^K, W^V; then R and
// the bins ([table row][query row] fp32), which the output staging tile overlays (at least
// 16 KB), and the barriers.
inline uint32_t layout(Params &p, bool ak, bool av, int ks, int vs) {
    const uint32_t qtile = (uint32_t)BM * D * 2;
    uint32_t off = 0;
    p.off_q = off;
    off += qtile;
    p.off_k = off;
    off += (uint32_t)ks * qtile;
    p.off_v = off;
    off += (uint32_t)vs * qtile;
    p.off_ak = off;
    if (ak) off += (uint32_t)p.npad_k * D * 2;
    p.off_av = off;
    if (av) off += (uint32_t)p.kpad_v * D * 2;
    p.off_r = off;
    p.off_stage = off;  // 1024-aligned: every size above is a multiple of 1024 bytes
    const uint32_t r0 = off;
    if (ak) off += (uint32_t)p.W * BM * 4;
    p.off_bins = off;
    if (av) off += (uint32_t)p.W * BM * 4;
    const uint32_t tile = (uint32_t)BM * D * 2;
    if (off - r0 < tile) off = r0 + tile;
    off = tc::round_up(off, 16);
    p.off_bar = off;
    off += (uint32_t)kNumBars * 8 + 16;
    p.kstages = ks;
    p.vstages = vs;
    return off + 1024;  // slack to align the base to 1024 bytes
}

}  // namespace sk

bool short_kernel_covers(const TcArgs &a) {
    if (a.mode != kShaw || a.d != sk::D || a.n > sk::kMaxTiles * sk::BN || a.n < 1) return false;
    if (a.aK || a.aV) {
        const int W = a.causal ? a.clip_k + 1 : 2 * a.clip_k + 1;
        if (W > sk::kMaxW) return false;
    }
    return true;
}

cudaError_t launch_short_bf16(const TcArgs &a, int *err_word, cudaStream_t s) {
    using namespace sk;
    if (!short_kernel_covers(a)) return cudaErrorNotSupported;
    const bool ak = a.aK != nullptr, av = a.aV != nullptr;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.BH = a.B * a.H;
    p.H = a.H;
    p.n = a.n;
    p.n_qtiles = (a.n + BM - 1) / BM;
    if ((long long)p.BH * p.n_qtiles > INT32_MAX) return cudaErrorNotSupported;
    p.num_units = p.BH * p.n_qtiles;
    p.scale_log2 = a.scale * kLog2e;
    p.kv_len = a.kv_len;
    p.err = err_word;
    p.out = a.out;
    p.clip_k = a.clip_k;
    p.W = (ak || av) ? (a.causal ? a.clip_k + 1 : 2 * a.clip_k + 1) : 1;
    p.npad_k = (int)tc::round_up((uint32_t)p.W, 16);
    p.kpad_v = p.npad_k;
    p.table_heads = a.ths != 0 ? 1 : 0;
    p.wait_limit = a.wait_limit > 0 ? a.wait_limit : 2000000000ll;
    p.withhold_q = a.withhold_q;
    if (p.BH == 0) return cudaSuccess;

    const tc::DeviceInfo di = tc::device_info();
    if (di.sms <= 0 || di.smem_optin <= 0 || di.smem_per_sm <= 0) return cudaErrorInvalidDevice;
    // two CTAs per SM: each takes half of the SM's shared memory (less the per-block
    // reservation) and at least a third of it, so that a third CTA never waits for TMEM
    const int64_t budget = (int64_t)di.smem_per_sm / 2 - di.smem_reserved;
    const int64_t floor3 = (int64_t)di.smem_per_sm / 3 + 1;
    // ring sizes, most stages first: a second K stage only helps when a unit has two key tiles
    const int two_tiles = p.n > BN;
    const int choices[4][2] = {{2, 2}, {2, 1}, {1, 2}, {1, 1}};
    uint32_t smem = 0;
    for (int c = 0; c < 4 && smem == 0; ++c) {
        if (!two_tiles && choices[c][0] == 2) continue;
        Params q = p;
        const uint32_t need = layout(q, ak, av, choices[c][0], choices[c][1]);
        if ((int64_t)need <= budget && (int64_t)need <= di.smem_optin) {
            p = q;
            smem = need;
        }
    }
    if (smem == 0) return cudaErrorNotSupported;
    if ((int64_t)smem < floor3) smem = (uint32_t)floor3;

    // TMA descriptors: q; k and v in 32-row boxes; k and v in whole-tile boxes; the tables;
    // the output (tile stores)
    CUtensorMap tm[8];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    if (!tc::make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !tc::make_map(&tm[1], a.k, d, n, BH, rs, hs, KB) ||
        !tc::make_map(&tm[2], a.v, d, n, BH, rs, hs, KB) || !tc::make_map(&tm[3], a.k, d, n, BH, rs, hs, BN) ||
        !tc::make_map(&tm[4], a.v, d, n, BH, rs, hs, BN) || !tc::make_map(&tm[7], a.out, d, n, BH, rs, hs, BM))
        return cudaErrorInvalidValue;
    tm[5] = tm[0];
    tm[6] = tm[0];
    const uint64_t rows = (uint64_t)(2 * a.clip_k + 1);
    const uint64_t Ht = p.table_heads ? (uint64_t)a.H : 1;
    const uint64_t ths_bytes = p.table_heads ? (uint64_t)a.ths * 2 : rows * d * 2;
    if (ak && !tc::make_map(&tm[5], a.aK, d, rows, Ht, rs, ths_bytes, (uint32_t)p.npad_k))
        return cudaErrorInvalidValue;
    if (av && !tc::make_map(&tm[6], a.aV, d, rows, Ht, rs, ths_bytes, (uint32_t)p.kpad_v))
        return cudaErrorInvalidValue;
    const int64_t slots = 2LL * di.sms;
    const int grid = (int)(p.num_units < slots ? p.num_units : slots);
    return a.causal ? sk::launch_terms<true>(ak, av, tm, p, smem, grid, s)
                    : sk::launch_terms<false>(ak, av, tm, p, smem, grid, s);
}

}  // namespace relattn
