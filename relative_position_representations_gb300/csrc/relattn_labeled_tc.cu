// Host side of the tensor-core kernel for labelled edges (relattn_labeled_tc.cuh): shared-memory
// layout, TMA descriptors, variant selection and launch. Head dimensions 64 and 128, bf16,
// up to 128 labels; the caller takes the SIMT kernel for anything else.
#include "relattn_labeled_tc.cuh"
#include "relattn_tc_launch.cuh"

namespace relattn {
namespace lbl {

template <int D, bool AK, bool AV, bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap (&tm)[7], const Params &p, uint32_t smem_bytes,
                           cudaStream_t s) {
    auto kern = relattn_labeled_tc_kernel<D, AK, AV, CAUSAL>;
    // opt in to the device's whole shared-memory budget once per device and variant, so that
    // later calls (including ones captured into a CUDA graph) only launch
    static bool opted[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const tc::DeviceInfo di = tc::device_info();
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opted[dev]) {
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

template <int D, bool CAUSAL>
cudaError_t launch_terms(bool ak, bool av, const CUtensorMap (&tm)[7], const Params &p,
                         uint32_t smem, cudaStream_t s) {
    if (ak && av) return launch_variant<D, true, true, CAUSAL>(tm, p, smem, s);
    if (ak) return launch_variant<D, true, false, CAUSAL>(tm, p, smem, s);
    if (av) return launch_variant<D, false, true, CAUSAL>(tm, p, smem, s);
    return launch_variant<D, false, false, CAUSAL>(tm, p, smem, s);
}

// Shared memory for `stages` K/V stages (the K ring takes stages - stages / 2, the V ring
// stages / 2); returns the bytes to request. TMA targets first (every size a multiple of
// 1024 bytes): the two Q buffers, the K and V rings, W^K, W^V; then the R rows, the two
// groups' value bins, the groups' exchange area (maxima by tile parity, row sums), barriers.
template <int D>
inline uint32_t layout(Params &p, bool ak, bool av, int stages) {
    const uint32_t q_bytes = (uint32_t)BM * D * 2;
    const uint32_t stage_bytes = (uint32_t)BN * D * 2;
    const int vs = stages / 2, ks = stages - vs;
    uint32_t off = 0;
    p.off_q[0] = off;
    off += q_bytes;
    p.off_q[1] = off;
    off += q_bytes;
    p.off_k = off;
    off += (uint32_t)ks * stage_bytes;
    p.off_v = off;
    off += (uint32_t)vs * stage_bytes;
    p.off_ak = off;
    if (ak) off += (uint32_t)p.npad_k * D * 2;
    p.off_av = off;
    if (av) off += (uint32_t)p.kpad_v * D * 2;
    p.off_r = off;
    if (ak) off += tc::round_up((uint32_t)BM * p.SR * 4, 16);
    p.off_beta[0] = off;
    if (av) off += tc::round_up((uint32_t)BM * p.SB * 4, 16);
    p.off_beta[1] = off;
    if (av) off += tc::round_up((uint32_t)BM * p.SB * 4, 16);
    p.off_x = off;
    off += 2 * 2 * BM * 4 + 2 * BM * 8;
    p.off_bar = off;
    off += (uint32_t)kNumBars * 8 + 16;
    // ceil(2^32 / n) for n >= 2 (a one-stage ring needs no reciprocal)
    auto mul = [](int n) { return n > 1 ? (uint32_t)((0x100000000ull + (uint64_t)n - 1) / (uint64_t)n) : 0u; };
    p.kstages = ks;
    p.vstages = vs;
    p.kmul = mul(ks);
    p.vmul = mul(vs);
    p.stage_bytes = stage_bytes;
    return off + 1024;  // slack to align the base to 1024 bytes
}

template <int D>
cudaError_t launch(const LabeledArgs &a, cudaStream_t s) {
    const bool ak = a.aK != nullptr, av = a.aV != nullptr;
    const int L = (ak || av) ? a.num_labels : 1;
    if (L < 1 || L > kMaxLabels) return cudaErrorNotSupported;
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.BH = a.B * a.H;
    p.H = a.H;
    p.n = a.n;
    p.n_qtiles = (a.n + BM - 1) / BM;
    if ((long long)p.BH * p.n_qtiles > INT32_MAX) return cudaErrorNotSupported;
    p.num_items = p.BH * p.n_qtiles;
    p.scale_log2 = a.scale * kLog2e;
    p.kv_len = a.kv_len;
    p.err = a.err;
    p.out = a.out;
    p.labels = a.labels;
    p.lbs = a.lbs;
    p.L = L;
    p.SR = L | 1;  // odd strides: the same label of the 32 rows of a warp lies in 32 banks
    p.SB = L | 1;
    p.npad_k = (int)tc::round_up((uint32_t)L, 16);
    p.kpad_v = p.npad_k;
    p.table_heads = a.ths != 0 ? 1 : 0;
    p.wait_limit = a.wait_limit > 0 ? a.wait_limit : 2000000000ll;
    p.lab_vec = (a.labels && reinterpret_cast<uintptr_t>(a.labels) % 16 == 0 && a.n % 16 == 0 &&
                 a.lbs % 16 == 0) ? 1 : 0;
    if (p.BH == 0) return cudaSuccess;
    if ((ak || av) && !a.labels) return cudaErrorInvalidValue;

    const tc::DeviceInfo di = tc::device_info();
    if (di.sms <= 0 || di.smem_optin <= 0) return cudaErrorInvalidDevice;
    const uint32_t fixed = layout<D>(p, ak, av, 0);
    int64_t st = ((int64_t)di.smem_optin - (int64_t)fixed) / ((int64_t)BN * D * 2);
    if (st > 2 * kMaxStages) st = 2 * kMaxStages;
    if (st < 2) return cudaErrorNotSupported;
    const uint32_t smem = layout<D>(p, ak, av, (int)st);
    if (smem > (uint32_t)di.smem_optin) return cudaErrorNotSupported;
    if (p.kstages < 1 || p.vstages < 1 || p.kstages > kMaxStages || p.vstages > kMaxStages)
        return cudaErrorNotSupported;

    // TMA descriptors: q; k and v in 32-row boxes; k and v in whole-tile boxes; the tables
    CUtensorMap tm[7];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    if (!tc::make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !tc::make_map(&tm[1], a.k, d, n, BH, rs, hs, KB) ||
        !tc::make_map(&tm[2], a.v, d, n, BH, rs, hs, KB) || !tc::make_map(&tm[3], a.k, d, n, BH, rs, hs, BN) ||
        !tc::make_map(&tm[4], a.v, d, n, BH, rs, hs, BN))
        return cudaErrorInvalidValue;
    tm[5] = tm[0];
    tm[6] = tm[0];
    const uint64_t Ht = p.table_heads ? (uint64_t)a.H : 1;
    const uint64_t ths_bytes = p.table_heads ? (uint64_t)a.ths * 2 : (uint64_t)L * d * 2;
    if (ak && !tc::make_map(&tm[5], a.aK, d, (uint64_t)L, Ht, rs, ths_bytes, (uint32_t)p.npad_k))
        return cudaErrorInvalidValue;
    if (av && !tc::make_map(&tm[6], a.aV, d, (uint64_t)L, Ht, rs, ths_bytes, (uint32_t)p.kpad_v))
        return cudaErrorInvalidValue;
    return a.causal ? launch_terms<D, true>(ak, av, tm, p, smem, s)
                    : launch_terms<D, false>(ak, av, tm, p, smem, s);
}

}  // namespace lbl

cudaError_t launch_labeled_tc(const LabeledArgs &a, cudaStream_t s) {
    if (!a.bf16) return cudaErrorNotSupported;
    if (a.d == 64) return lbl::launch<64>(a, s);
    if (a.d == 128) return lbl::launch<128>(a, s);
    return cudaErrorNotSupported;
}

}  // namespace relattn
