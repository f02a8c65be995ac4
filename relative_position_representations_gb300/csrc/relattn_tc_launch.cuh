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
    int smem_optin = 0;
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
    }
    return cache[dev];
}

inline uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int D, bool AK, bool AV, bool T5, bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap (&tm)[6], const Params &p, uint32_t smem_bytes, int grid,
                           cudaStream_t s) {
    auto kern = relattn_tc_kernel<D, AK, AV, T5, CAUSAL>;
    // Opt in to the device's whole shared-memory budget once per device and variant, so
    // that later calls (including ones captured into a CUDA graph) only launch.
    static bool opted[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opted[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     device_info().smem_optin);
            if (e != cudaSuccess) return e;
            opted[dev] = true;
        }
    }
    kern<<<grid, kThreads, smem_bytes, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], tm[5], p);
    return cudaGetLastError();
}

template <int D, bool T5, bool CAUSAL>
cudaError_t launch_terms(bool ak, bool av, const CUtensorMap (&tm)[6], const Params &p,
                         uint32_t smem, int grid, cudaStream_t s) {
    if constexpr (T5) {
        return launch_variant<D, false, false, true, CAUSAL>(tm, p, smem, grid, s);
    } else {
        if (ak && av) return launch_variant<D, true, true, false, CAUSAL>(tm, p, smem, grid, s);
        if (ak) return launch_variant<D, true, false, false, CAUSAL>(tm, p, smem, grid, s);
        if (av) return launch_variant<D, false, true, false, CAUSAL>(tm, p, smem, grid, s);
        return launch_variant<D, false, false, false, CAUSAL>(tm, p, smem, grid, s);
    }
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
    p.num_tiles = p.BH * p.n_qtiles;
    p.scale_log2 = a.scale * kLog2e;
    p.kv_len = a.kv_len;
    p.err = err_word;
    p.clip_k = a.clip_k;
    p.W = 1;
    if (ak || av) {
        p.W = a.causal ? a.clip_k + 1 : 2 * a.clip_k + 1;
        if (p.W > 128) return cudaErrorNotSupported;
    }
    p.SR = p.W + (p.W & 1);
    p.npad_k = (int)round_up((uint32_t)p.W, 16);
    p.kpad_v = p.npad_k;
    p.table_heads = a.ths != 0 ? 1 : 0;
    p.bias = a.bias;
    if (t5mode) {
        p.t5 = *t5;
        p.t5_R = t5->sat;
    }
    if (p.num_tiles == 0) return cudaSuccess;

    const DeviceInfo di = device_info();
    if (di.sms <= 0 || di.smem_optin <= 0) return cudaErrorInvalidDevice;
    // ---- shared-memory layout (offsets from a 1024-aligned base)
    const uint32_t tile_bytes = (uint32_t)BM * D * 2;
    uint32_t fixed = tile_bytes;                        // Q
    fixed += (uint32_t)BM * BN * 2;                     // P / bins / output staging
    if (ak) fixed += (uint32_t)p.npad_k * D * 2;        // W^K rows
    if (av) fixed += (uint32_t)p.kpad_v * D * 2;        // W^V rows
    if (ak) fixed += round_up((uint32_t)BM * p.SR * 4, 1024);
    if (av) fixed += round_up((uint32_t)BM * p.SR * 4, 1024);
    if (t5mode) fixed += round_up((uint32_t)(2 * p.t5_R + 1) * 4, 1024);
    fixed += round_up((uint32_t)kNumBars * 8 + 16, 1024);
    const uint32_t slack = 1024;
    const int64_t room = (int64_t)di.smem_optin - (int64_t)fixed - slack;
    int stages = (int)(room / (int64_t)tile_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorNotSupported;
    p.stages = stages;
    p.stage_bytes = tile_bytes;
    uint32_t off = 0;
    p.off_q = off;    off += tile_bytes;
    p.off_kv = off;   off += (uint32_t)stages * tile_bytes;
    p.off_p = off;    off += (uint32_t)BM * BN * 2;
    p.off_ak = off;   if (ak) off += (uint32_t)p.npad_k * D * 2;
    p.off_av = off;   if (av) off += (uint32_t)p.kpad_v * D * 2;
    p.off_r = off;    if (ak) off += round_up((uint32_t)BM * p.SR * 4, 1024);
    p.off_beta = off; if (av) off += round_up((uint32_t)BM * p.SR * 4, 1024);
    p.off_t5 = off;   if (t5mode) off += round_up((uint32_t)(2 * p.t5_R + 1) * 4, 1024);
    p.off_bar = off;  off += round_up((uint32_t)kNumBars * 8 + 16, 1024);
    const uint32_t smem_bytes = off + slack;
    if (smem_bytes > (uint32_t)di.smem_optin) return cudaErrorNotSupported;

    // ---- TMA descriptors
    CUtensorMap tm[6];
    const uint64_t d = (uint64_t)D, n = (uint64_t)a.n, BH = (uint64_t)p.BH;
    const uint64_t rs = d * 2, hs = n * d * 2;
    if (!make_map(&tm[0], a.q, d, n, BH, rs, hs, BM) || !make_map(&tm[1], a.k, d, n, BH, rs, hs, BN) ||
        !make_map(&tm[2], a.v, d, n, BH, rs, hs, BN) || !make_map(&tm[3], a.out, d, n, BH, rs, hs, BM))
        return cudaErrorInvalidValue;
    tm[4] = tm[0];
    tm[5] = tm[0];
    const uint64_t rows = (uint64_t)(2 * a.clip_k + 1);
    const uint64_t Ht = p.table_heads ? (uint64_t)a.H : 1;
    const uint64_t ths_bytes = p.table_heads ? (uint64_t)a.ths * 2 : rows * d * 2;
    if (ak && !make_map(&tm[4], a.aK, d, rows, Ht, rs, ths_bytes, (uint32_t)p.npad_k))
        return cudaErrorInvalidValue;
    if (av && !make_map(&tm[5], a.aV, d, rows, Ht, rs, ths_bytes, (uint32_t)p.kpad_v))
        return cudaErrorInvalidValue;

    const int grid = p.num_tiles < di.sms ? p.num_tiles : di.sms;
    if (a.causal) {
        return t5mode ? launch_terms<D, true, true>(ak, av, tm, p, smem_bytes, grid, s)
                      : launch_terms<D, false, true>(ak, av, tm, p, smem_bytes, grid, s);
    }
    return t5mode ? launch_terms<D, true, false>(ak, av, tm, p, smem_bytes, grid, s)
                  : launch_terms<D, false, false>(ak, av, tm, p, smem_bytes, grid, s);
}

}  // namespace tc
}  // namespace relattn
