// Public C ABI of librelattn.so (declared in include/relattn.h): argument validation,
// dispatch to the fp32 SIMT path or the bf16 tcgen05 path, device status word.
#include <cstdint>
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/relattn.h"
#include "relattn_internal.h"

namespace {

// device status word: bounded waits that run out record RELATTN_ERR_TIMEOUT here
__device__ int g_status_word;

int *status_word_for_current_device() {
    static int *addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int *>(p);
    }
    return addr[dev];
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// device scratch of relattn_decode_fwd_noalloc: part of the module image, never allocated
constexpr unsigned long long kStaticScratchBytes = 4ull << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// its address on the current device, looked up once per device with that device current
void *static_scratch_for_current_device() {
    static void *addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

// compute capability of the current device (major*10 + minor), or -1
int current_cc() {
    int dev = 0, ma = 0, mi = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return -1;
    return ma * 10 + mi;
}

relattn_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return RELATTN_OK;
    if (e == cudaErrorNotSupported) return RELATTN_ERR_UNSUPPORTED;
    cudaGetLastError();  // do not leave a launch-configuration error sticky for the caller
    return RELATTN_ERR_CUDA;
}

bool shapes_ok(int B, int H, int n, int d) {
    if (B < 1 || H < 1 || n < 1 || d < 1) return false;
    const long long total = (long long)B * H * n;
    return total <= (1LL << 31) - 1 && (long long)B * H <= (1LL << 31) - 1;
}

// common checks of q, k, v, out
relattn_status_t check_qkv(const void *q, const void *k, const void *v, const void *out, int B,
                           int H, int n, int d, int dtype) {
    if (!q || !k || !v || !out) return RELATTN_ERR_INVALID_ARG;
    if (!shapes_ok(B, H, n, d)) return RELATTN_ERR_INVALID_ARG;
    if (out == q || out == k || out == v) return RELATTN_ERR_INVALID_ARG;
    if (dtype == RELATTN_BF16) {
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
            return RELATTN_ERR_INVALID_ARG;
        if (d != 64 && d != 128) return RELATTN_ERR_UNSUPPORTED;
    } else if (dtype == RELATTN_F32) {
        if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(out, 4))
            return RELATTN_ERR_INVALID_ARG;
        if (d > 128) return RELATTN_ERR_UNSUPPORTED;
    } else {
        return RELATTN_ERR_INVALID_ARG;
    }
    return RELATTN_OK;
}

// bound of the fused kernel's device waits (SM clock cycles) and the timeout-test hook,
// read at each launch
std::atomic<long long> g_wait_limit{2000000000ll};
std::atomic<int> g_withhold_q{0};
std::atomic<int> g_short_kernel{1};
std::atomic<int> g_bwd_tensor_cores{1};

relattn_status_t dispatch_bf16(const relattn::TcArgs &args, const relattn::T5Buckets *t5,
                               cudaStream_t s) {
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    int *err = status_word_for_current_device();
    if (!err) return RELATTN_ERR_CUDA;
    relattn::TcArgs a = args;
    a.wait_limit = g_wait_limit.load();
    a.withhold_q = g_withhold_q.load();
    if (g_short_kernel.load() && relattn::short_kernel_covers(a)) {
        const cudaError_t e = relattn::launch_short_bf16(a, err, s);
        if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    const cudaError_t e = a.d == 64 ? relattn::launch_tc_bf16_d64(a, t5, err, s)
                                    : relattn::launch_tc_bf16_d128(a, t5, err, s);
    return from_cuda(e);
}

// Forward with a scalar bias per offset (T5 buckets, ALiBi or a clipped per-offset table):
// shared checks, then the fp32 SIMT path or the bf16 tcgen05 path.
relattn_status_t scalar_bias_fwd(const void *q, const void *k, const void *v, const float *bias,
                                 int kind, int radius, long long head_stride,
                                 const relattn::T5Buckets *t5, int causal, float scale,
                                 const int *kv_len, int B, int H, int n, int d, int dtype,
                                 void *out, relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, out, B, H, n, d, dtype);
    if (st != RELATTN_OK) return st;
    if (!bias || !aligned(bias, 4)) return RELATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    relattn::T5Buckets none{};
    const relattn::T5Buckets *tb = t5 ? t5 : &none;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == RELATTN_F32) {
        relattn::SimtArgs a{};
        a.q = static_cast<const float *>(q);
        a.k = static_cast<const float *>(k);
        a.v = static_cast<const float *>(v);
        a.causal = causal;
        a.scale = scale;
        a.kv_len = kv_len;
        a.bias = bias;
        a.bias_kind = kind;
        a.bias_R = radius;
        a.bias_hs = head_stride;
        a.B = B; a.H = H; a.n = n; a.d = d;
        a.out = static_cast<float *>(out);
        return from_cuda(relattn::launch_simt_f32(a, tb, s));
    }
    relattn::TcArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.bias = bias;
    a.bias_kind = kind;
    a.bias_R = radius;
    a.bias_hs = head_stride;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.out = out;
    a.mode = relattn::kT5;
    return dispatch_bf16(a, tb, s);
}

}  // namespace

extern "C" {

relattn_status_t relattn_fwd(const void *q, const void *k, const void *v, const void *aK,
                             const void *aV, long long table_head_stride, int clip_k, int causal,
                             float scale, const int *kv_len, int B, int H, int n, int d, int dtype,
                             void *out, relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, out, B, H, n, d, dtype);
    if (st != RELATTN_OK) return st;
    if (clip_k < 0 || (causal != 0 && causal != 1)) return RELATTN_ERR_INVALID_ARG;
    if (clip_k > (1 << 20)) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    if (aK || aV) {
        const long long rows_d = (2LL * clip_k + 1) * d;
        if (table_head_stride != 0 && table_head_stride < rows_d) return RELATTN_ERR_INVALID_ARG;
        if (out == aK || out == aV) return RELATTN_ERR_INVALID_ARG;
        const uintptr_t al = dtype == RELATTN_BF16 ? 16 : 4;
        if ((aK && !aligned(aK, al)) || (aV && !aligned(aV, al))) return RELATTN_ERR_INVALID_ARG;
        if (dtype == RELATTN_BF16 && (table_head_stride % 8) != 0) return RELATTN_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == RELATTN_F32) {
        relattn::SimtArgs a{};
        a.q = static_cast<const float *>(q);
        a.k = static_cast<const float *>(k);
        a.v = static_cast<const float *>(v);
        a.aK = static_cast<const float *>(aK);
        a.aV = static_cast<const float *>(aV);
        a.ths = table_head_stride;
        a.clip_k = clip_k;
        a.causal = causal;
        a.scale = scale;
        a.kv_len = kv_len;
        a.bias = nullptr;
        a.B = B; a.H = H; a.n = n; a.d = d;
        a.out = static_cast<float *>(out);
        return from_cuda(relattn::launch_simt_f32(a, nullptr, s));
    }
    relattn::TcArgs a{};
    a.q = q; a.k = k; a.v = v; a.aK = aK; a.aV = aV;
    a.ths = table_head_stride;
    a.clip_k = clip_k;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.bias = nullptr;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.out = out;
    a.mode = relattn::kShaw;
    return dispatch_bf16(a, nullptr, s);
}

relattn_status_t relattn_decode_workspace_size(int B, int H, int T, int d,
                                               unsigned long long *bytes) {
    if (!bytes || !shapes_ok(B, H, T, d)) return RELATTN_ERR_INVALID_ARG;
    *bytes = relattn::decode_workspace_bytes(B, H, T, d);
    return RELATTN_OK;
}

relattn_status_t relattn_decode_fwd(const void *q, const void *k_cache, const void *v_cache,
                                    const void *aK, const void *aV, long long table_head_stride,
                                    int clip_k, float scale, const int *cache_len, int B, int H,
                                    int T, int d, void *workspace,
                                    unsigned long long workspace_bytes, void *out,
                                    relattn_stream_t stream) {
    if (!q || !k_cache || !v_cache || !out || !cache_len) return RELATTN_ERR_INVALID_ARG;
    if (!shapes_ok(B, H, T, d)) return RELATTN_ERR_INVALID_ARG;
    if (out == q || out == k_cache || out == v_cache || out == aK || out == aV)
        return RELATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(cache_len, 4) || (workspace && !aligned(workspace, 16)))
        return RELATTN_ERR_INVALID_ARG;
    if (clip_k < 0 || clip_k > (1 << 20)) return RELATTN_ERR_INVALID_ARG;
    if (aK || aV) {
        const long long rows_d = (2LL * clip_k + 1) * d;
        if (table_head_stride != 0 && table_head_stride < rows_d) return RELATTN_ERR_INVALID_ARG;
        if ((aK && !aligned(aK, 16)) || (aV && !aligned(aV, 16))) return RELATTN_ERR_INVALID_ARG;
        if ((table_head_stride % 8) != 0) return RELATTN_ERR_INVALID_ARG;
    }
    if (d != 64 && d != 128) return RELATTN_ERR_UNSUPPORTED;
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    relattn::DecodeArgs a{};
    a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.aK = aK; a.aV = aV;
    a.ths = table_head_stride;
    a.clip_k = clip_k;
    a.scale = scale;
    a.cache_len = cache_len;
    a.B = B; a.H = H; a.T = T; a.d = d;
    a.out = out;
    a.workspace = workspace;
    a.workspace_bytes = workspace ? workspace_bytes : 0;
    return from_cuda(relattn::launch_decode_bf16(a, reinterpret_cast<cudaStream_t>(stream)));
}

relattn_status_t relattn_labeled_fwd(const void *q, const void *k, const void *v,
                                     const void *aK, const void *aV, long long table_head_stride,
                                     int num_labels, const unsigned char *labels,
                                     long long label_batch_stride, int causal, float scale,
                                     const int *kv_len, int B, int H, int n, int d, int dtype,
                                     void *out, relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, out, B, H, n, d, dtype);
    // this path takes any head dimension up to 128 whose rows are whole 16-byte vectors
    if (st != RELATTN_OK && st != RELATTN_ERR_UNSUPPORTED) return st;
    if (!shapes_ok(B, H, n, d)) return RELATTN_ERR_INVALID_ARG;
    const int vec = dtype == RELATTN_BF16 ? 8 : 4;
    if (d > 128 || d % vec != 0) return RELATTN_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return RELATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    if (aK || aV) {
        if (num_labels < 1 || num_labels > 256 || !labels) return RELATTN_ERR_INVALID_ARG;
        if ((aK && !aligned(aK, 16)) || (aV && !aligned(aV, 16))) return RELATTN_ERR_INVALID_ARG;
        if (table_head_stride != 0 &&
            (table_head_stride < (long long)num_labels * d || table_head_stride % vec != 0))
            return RELATTN_ERR_INVALID_ARG;
        if (label_batch_stride != 0 && label_batch_stride < (long long)n * n)
            return RELATTN_ERR_INVALID_ARG;
    }
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    int *err = status_word_for_current_device();
    if (!err) return RELATTN_ERR_CUDA;
    relattn::LabeledArgs a{};
    a.q = q; a.k = k; a.v = v; a.aK = aK; a.aV = aV;
    a.ths = table_head_stride;
    a.num_labels = (aK || aV) ? num_labels : 0;
    a.labels = labels;
    a.lbs = label_batch_stride;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.bf16 = dtype == RELATTN_BF16 ? 1 : 0;
    a.out = out;
    a.err = err;
    a.wait_limit = g_wait_limit.load();
    // bf16 with d = 64 or 128 runs on the tensor cores when the kernel fits the shapes (at
    // most 128 labels); the SIMT kernel takes everything else
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (a.bf16 && (d == 64 || d == 128)) {
        const cudaError_t e = relattn::launch_labeled_tc(a, cs);
        if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    return from_cuda(relattn::launch_labeled(a, cs));
}

relattn_status_t relattn_txl_fwd(const void *q, const void *k, const void *v, const void *rel,
                                 const void *u, const void *vb, int shared, int causal, float scale,
                                 const int *kv_len, int B, int H, int n, int d, int dtype,
                                 void *out, relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, out, B, H, n, d, dtype);
    // this path takes any head dimension up to 128 whose rows are whole 16-byte vectors
    if (st != RELATTN_OK && st != RELATTN_ERR_UNSUPPORTED) return st;
    if (!shapes_ok(B, H, n, d)) return RELATTN_ERR_INVALID_ARG;
    if ((long long)H * (2LL * n - 1) * d > (1LL << 40)) return RELATTN_ERR_INVALID_ARG;
    const int vec = dtype == RELATTN_BF16 ? 8 : 4;
    if (d > 128 || d % vec != 0) return RELATTN_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return RELATTN_ERR_INVALID_ARG;
    if (!rel || !u || !vb || !aligned(rel, 16)) return RELATTN_ERR_INVALID_ARG;
    const uintptr_t el = dtype == RELATTN_BF16 ? 2 : 4;
    if (!aligned(u, el) || !aligned(vb, el)) return RELATTN_ERR_INVALID_ARG;
    if ((shared != 0 && shared != 1) || (causal != 0 && causal != 1)) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    relattn::TxlArgs a{};
    a.q = q; a.k = k; a.v = v; a.rel = rel; a.u = u; a.vb = vb;
    a.shared = shared;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.bf16 = dtype == RELATTN_BF16 ? 1 : 0;
    a.out = out;
    a.wait_limit = g_wait_limit.load();
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (relattn::txl_tc_covers(a)) {
        a.err = status_word_for_current_device();
        if (!a.err) return RELATTN_ERR_CUDA;
        const cudaError_t e = relattn::launch_txl_tc(a, s);
        if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    return from_cuda(relattn::launch_txl(a, s));
}

relattn_status_t relattn_decode_fwd_noalloc(const void *q, const void *k_cache,
                                            const void *v_cache, const void *aK, const void *aV,
                                            long long table_head_stride, int clip_k, float scale,
                                            const int *cache_len, int B, int H, int T, int d,
                                            void *out, relattn_stream_t stream) {
    void *ws = static_scratch_for_current_device();
    if (!ws) return RELATTN_ERR_CUDA;
    return relattn_decode_fwd(q, k_cache, v_cache, aK, aV, table_head_stride, clip_k, scale,
                              cache_len, B, H, T, d, ws, kStaticScratchBytes, out, stream);
}

relattn_status_t relattn_labeled_bwd_workspace_size(int B, int H, int n, int num_labels,
                                                  unsigned long long *bytes) {
    if (!bytes || !shapes_ok(B, H, n, 1) || num_labels < 1 || num_labels > 256)
        return RELATTN_ERR_INVALID_ARG;
    *bytes = relattn::bwd_simt_workspace_bytes(B, H, n, num_labels);
    return RELATTN_OK;
}

relattn_status_t relattn_labeled_bwd(const void *q, const void *k, const void *v, const void *aK,
                                     const void *aV, long long table_head_stride, int num_labels,
                                     const unsigned char *labels, long long label_batch_stride,
                                     int causal, float scale, const int *kv_len, int B, int H,
                                     int n, int d, int dtype, const void *dout, float *dq,
                                     float *dk, float *dv, float *daK, float *daV,
                                     void *workspace, unsigned long long workspace_bytes,
                                     relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, dq, B, H, n, d, dtype);
    if (st != RELATTN_OK && st != RELATTN_ERR_UNSUPPORTED) return st;
    if (!dout || !dk || !dv || !workspace) return RELATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    const uintptr_t al = dtype == RELATTN_BF16 ? 2 : 4;
    if (!aligned(dout, al) || !aligned(dk, 4) || !aligned(dv, 4) || !aligned(workspace, 4))
        return RELATTN_ERR_INVALID_ARG;
    if (num_labels < 1 || num_labels > 256 || !labels) return RELATTN_ERR_INVALID_ARG;
    if (label_batch_stride < 0 || (label_batch_stride != 0 && label_batch_stride < (long long)n * n))
        return RELATTN_ERR_INVALID_ARG;
    if ((aK && !daK) || (aV && !daV)) return RELATTN_ERR_INVALID_ARG;
    if (aK || aV) {
        if (table_head_stride < 0 ||
            (table_head_stride != 0 && table_head_stride < (long long)num_labels * d))
            return RELATTN_ERR_INVALID_ARG;
        if ((aK && !aligned(aK, al)) || (aV && !aligned(aV, al)) || (daK && !aligned(daK, 4)) ||
            (daV && !aligned(daV, 4)))
            return RELATTN_ERR_INVALID_ARG;
    }
    if (d > 128) return RELATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < relattn::bwd_simt_workspace_bytes(B, H, n, num_labels))
        return RELATTN_ERR_INVALID_ARG;
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    relattn::BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.aK = aK; a.aV = aV; a.dout = dout;
    a.ths = table_head_stride;
    a.clip_k = 0;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.bf16 = dtype == RELATTN_BF16 ? 1 : 0;
    a.dq = dq; a.dk = dk; a.dv = dv; a.daK = daK; a.daV = daV;
    a.workspace = workspace;
    a.labels = labels;
    a.lbs = label_batch_stride;
    a.num_labels = num_labels;
    a.err = status_word_for_current_device();
    if (!a.err) return RELATTN_ERR_CUDA;
    return from_cuda(relattn::launch_bwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

relattn_status_t relattn_scalar_bias_bwd_workspace_size(int B, int H, int n,
                                                      unsigned long long *bytes) {
    if (!bytes || B < 0 || H < 0 || n < 0) return RELATTN_ERR_INVALID_ARG;
    *bytes = relattn::bias_bwd_workspace_bytes(B, H, n);
    return RELATTN_OK;
}

relattn_status_t relattn_scalar_bias_bwd(const void *q, const void *k, const void *v,
                                         const void *dout, int kind, const float *bias,
                                         int num_buckets, int max_distance, int bidirectional,
                                         int radius, long long bias_head_stride, int causal,
                                         float scale, const int *kv_len, int B, int H, int n,
                                         int d, int dtype, float *dq, float *dk, float *dv,
                                         float *dbias, void *workspace,
                                         unsigned long long workspace_bytes,
                                         relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, dq, B, H, n, d, dtype);
    if (st != RELATTN_OK && st != RELATTN_ERR_UNSUPPORTED) return st;
    if (!dout || !dk || !dv || !dbias || !bias || !workspace) return RELATTN_ERR_INVALID_ARG;
    const uintptr_t al = dtype == RELATTN_BF16 ? 2 : 4;
    if (!aligned(dout, al) || !aligned(dk, 4) || !aligned(dv, 4) || !aligned(dbias, 4) ||
        !aligned(bias, 4) || !aligned(workspace, 4))
        return RELATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    relattn::T5Buckets t5{};
    if (kind == relattn::kBiasBuckets) {
        if (bidirectional != 0 && bidirectional != 1) return RELATTN_ERR_INVALID_ARG;
        if (!relattn::t5_make_buckets(num_buckets, max_distance, bidirectional, &t5))
            return RELATTN_ERR_INVALID_ARG;
    } else if (kind == relattn::kBiasTable) {
        if (radius < 0 || radius > (1 << 20)) return RELATTN_ERR_INVALID_ARG;
        if (bias_head_stride < 0 || (bias_head_stride != 0 && bias_head_stride < 2LL * radius + 1))
            return RELATTN_ERR_INVALID_ARG;
    } else if (kind != relattn::kBiasAlibi) {
        return RELATTN_ERR_INVALID_ARG;
    }
    if (d > 128 || n > relattn::kBiasBwdMaxN) return RELATTN_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535) return RELATTN_ERR_UNSUPPORTED;  // sequence-heads on grid y
    if (workspace_bytes < relattn::bias_bwd_workspace_bytes(B, H, n)) return RELATTN_ERR_INVALID_ARG;
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    relattn::BiasBwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.dout = dout;
    a.bias = bias;
    a.kind = kind;
    a.num_buckets = num_buckets;
    a.radius = radius;
    a.head_stride = bias_head_stride;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.bf16 = dtype == RELATTN_BF16 ? 1 : 0;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dbias = dbias;
    a.workspace = workspace;
    return from_cuda(relattn::launch_bias_bwd(a, kind == relattn::kBiasBuckets ? &t5 : nullptr,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

relattn_status_t relattn_bwd_workspace_size(int B, int H, int n, int d, int clip_k,
                                            unsigned long long *bytes) {
    if (!bytes || !shapes_ok(B, H, n, d) || clip_k < 0 || clip_k > (1 << 20))
        return RELATTN_ERR_INVALID_ARG;
    *bytes = relattn::bwd_workspace_bytes(B, H, n, clip_k);
    return RELATTN_OK;
}

relattn_status_t relattn_bwd(const void *q, const void *k, const void *v, const void *aK,
                             const void *aV, long long table_head_stride, int clip_k, int causal,
                             float scale, const int *kv_len, int B, int H, int n, int d,
                             int dtype, const void *dout, float *dq, float *dk, float *dv,
                             float *daK, float *daV, void *workspace,
                             unsigned long long workspace_bytes, relattn_stream_t stream) {
    relattn_status_t st = check_qkv(q, k, v, dq, B, H, n, d, dtype);
    if (st != RELATTN_OK && st != RELATTN_ERR_UNSUPPORTED) return st;
    if (!dout || !dk || !dv || !workspace) return RELATTN_ERR_INVALID_ARG;
    if (d > 128) return RELATTN_ERR_UNSUPPORTED;
    if (clip_k < 0 || clip_k > (1 << 20) || (causal != 0 && causal != 1)) return RELATTN_ERR_INVALID_ARG;
    if (kv_len && !aligned(kv_len, 4)) return RELATTN_ERR_INVALID_ARG;
    const uintptr_t al = dtype == RELATTN_BF16 ? 2 : 4;
    if (!aligned(dout, al) || !aligned(dk, 4) || !aligned(dv, 4) || !aligned(workspace, 4))
        return RELATTN_ERR_INVALID_ARG;
    if ((aK && !daK) || (aV && !daV)) return RELATTN_ERR_INVALID_ARG;
    if (aK || aV) {
        const long long rows_d = (2LL * clip_k + 1) * d;
        if (table_head_stride != 0 && table_head_stride < rows_d) return RELATTN_ERR_INVALID_ARG;
        if ((daK && !aligned(daK, 4)) || (daV && !aligned(daV, 4))) return RELATTN_ERR_INVALID_ARG;
    }
    if (workspace_bytes < relattn::bwd_workspace_bytes(B, H, n, clip_k)) return RELATTN_ERR_INVALID_ARG;
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    relattn::BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.aK = aK; a.aV = aV; a.dout = dout;
    a.ths = table_head_stride;
    a.clip_k = clip_k;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.B = B; a.H = H; a.n = n; a.d = d;
    a.bf16 = dtype == RELATTN_BF16 ? 1 : 0;
    a.dq = dq; a.dk = dk; a.dv = dv; a.daK = daK; a.daV = daV;
    a.workspace = workspace;
    a.wait_limit = g_wait_limit.load();
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (g_bwd_tensor_cores.load() && relattn::bwd_tc_covers(a)) {
        a.err = status_word_for_current_device();
        if (!a.err) return RELATTN_ERR_CUDA;
        const cudaError_t e = relattn::launch_bwd_tc(a, s);
        if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    return from_cuda(relattn::launch_bwd(a, s));
}

relattn_status_t relattn_t5bias_fwd(const void *q, const void *k, const void *v,
                                    const float *bias, int num_buckets, int max_distance,
                                    int bidirectional, int causal, float scale,
                                    const int *kv_len, int B, int H, int n, int d, int dtype,
                                    void *out, relattn_stream_t stream) {
    if (bidirectional != 0 && bidirectional != 1) return RELATTN_ERR_INVALID_ARG;
    relattn::T5Buckets t5{};
    if (!relattn::t5_make_buckets(num_buckets, max_distance, bidirectional, &t5))
        return RELATTN_ERR_INVALID_ARG;
    return scalar_bias_fwd(q, k, v, bias, relattn::kBiasBuckets, 0, 0, &t5, causal, scale,
                           kv_len, B, H, n, d, dtype, out, stream);
}

relattn_status_t relattn_alibi_fwd(const void *q, const void *k, const void *v,
                                   const float *slopes, int causal, float scale,
                                   const int *kv_len, int B, int H, int n, int d, int dtype,
                                   void *out, relattn_stream_t stream) {
    return scalar_bias_fwd(q, k, v, slopes, relattn::kBiasAlibi, 0, 0, nullptr, causal, scale,
                           kv_len, B, H, n, d, dtype, out, stream);
}

relattn_status_t relattn_offset_bias_fwd(const void *q, const void *k, const void *v,
                                         const float *table, long long table_head_stride,
                                         int radius, int causal, float scale,
                                         const int *kv_len, int B, int H, int n, int d,
                                         int dtype, void *out, relattn_stream_t stream) {
    if (radius < 0 || radius > (1 << 20)) return RELATTN_ERR_INVALID_ARG;
    if (table_head_stride != 0 && table_head_stride < 2LL * radius + 1) return RELATTN_ERR_INVALID_ARG;
    return scalar_bias_fwd(q, k, v, table, relattn::kBiasTable, radius, table_head_stride,
                           nullptr, causal, scale, kv_len, B, H, n, d, dtype, out, stream);
}

relattn_status_t relattn_labels(int kind, int clip_k, int num_buckets, int max_distance,
                                int bidirectional, int n_q, int n_k, int *labels,
                                relattn_stream_t stream) {
    if (!labels || !aligned(labels, 4) || n_q < 0 || n_k < 0) return RELATTN_ERR_INVALID_ARG;
    if ((long long)n_q * n_k > (1LL << 40)) return RELATTN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (kind == 0) {
        if (clip_k < 0) return RELATTN_ERR_INVALID_ARG;
        return from_cuda(relattn::launch_labels(0, clip_k, nullptr, n_q, n_k, labels, s));
    }
    if (kind == 1) {
        relattn::T5Buckets t5{};
        if (!relattn::t5_make_buckets(num_buckets, max_distance, bidirectional ? 1 : 0, &t5))
            return RELATTN_ERR_INVALID_ARG;
        return from_cuda(relattn::launch_labels(1, 0, &t5, n_q, n_k, labels, s));
    }
    return RELATTN_ERR_INVALID_ARG;
}

relattn_status_t relattn_t5_thresholds(int num_buckets, int max_distance, int bidirectional,
                                       int *thresholds, int capacity, int *count) {
    if (!count) return RELATTN_ERR_INVALID_ARG;
    relattn::T5Buckets t5{};
    if (!relattn::t5_make_buckets(num_buckets, max_distance, bidirectional ? 1 : 0, &t5))
        return RELATTN_ERR_INVALID_ARG;
    *count = t5.nthr;
    if (t5.nthr > 0 && (!thresholds || capacity < t5.nthr)) return RELATTN_ERR_INVALID_ARG;
    for (int i = 0; i < t5.nthr; ++i) thresholds[i] = t5.thr[i];
    return RELATTN_OK;
}

relattn_status_t relattn_get_device_error(relattn_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return RELATTN_ERR_CUDA;
    int *w = status_word_for_current_device();
    if (!w) return RELATTN_ERR_CUDA;
    int host = 0;
    if (cudaMemcpyAsync(&host, w, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RELATTN_ERR_CUDA;
    if (cudaMemsetAsync(w, 0, sizeof(int), s) != cudaSuccess) return RELATTN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RELATTN_ERR_CUDA;
    return host == 0 ? RELATTN_OK : static_cast<relattn_status_t>(host);
}

const char *relattn_status_string(relattn_status_t s) {
    switch (s) {
        case RELATTN_OK: return "ok";
        case RELATTN_ERR_INVALID_ARG: return "invalid argument";
        case RELATTN_ERR_UNSUPPORTED: return "unsupported combination";
        case RELATTN_ERR_CUDA: return "CUDA error";
        case RELATTN_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

relattn_status_t relattn_set_wait_limit(long long cycles) {
    if (cycles < 1000 || cycles > (1ll << 40)) return RELATTN_ERR_INVALID_ARG;
    g_wait_limit.store(cycles);
    return RELATTN_OK;
}

relattn_status_t relattn_debug_withhold_first_load(int on) {
    if (on != 0 && on != 1) return RELATTN_ERR_INVALID_ARG;
    g_withhold_q.store(on);
    return RELATTN_OK;
}

relattn_status_t relattn_sinusoid_table(int n, int d_model, int dtype, void *out,
                                        relattn_stream_t stream) {
    if (!out || n < 1 || n > (1 << 28) || d_model < 2 || d_model > (1 << 16) || (d_model & 1))
        return RELATTN_ERR_INVALID_ARG;
    if (dtype != RELATTN_BF16 && dtype != RELATTN_F32) return RELATTN_ERR_INVALID_ARG;
    if (!aligned(out, dtype == RELATTN_BF16 ? 2 : 4)) return RELATTN_ERR_INVALID_ARG;
    const int cc = current_cc();
    if (cc < 0) return RELATTN_ERR_CUDA;
    if (cc != 103) return RELATTN_ERR_UNSUPPORTED;  // built for sm_103a only
    return from_cuda(relattn::launch_sinusoid(n, d_model, dtype == RELATTN_BF16 ? 1 : 0, out,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

relattn_status_t relattn_set_short_kernel(int on) {
    if (on != 0 && on != 1) return RELATTN_ERR_INVALID_ARG;
    g_short_kernel.store(on);
    return RELATTN_OK;
}

relattn_status_t relattn_set_bwd_tensor_cores(int on) {
    if (on != 0 && on != 1) return RELATTN_ERR_INVALID_ARG;
    g_bwd_tensor_cores.store(on);
    return RELATTN_OK;
}

int relattn_version(void) { return 102; }

}  // extern "C"
