// Internal declarations shared by the translation units of librelattn.so.
// Nothing here is part of the public C ABI (include/relattn.h).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace relattn {

constexpr int kMaxT5Thresholds = 128;

// Exact T5 bucketing parameters; thr[m] is the first distance a of bucket exact+1+m.
struct T5Buckets {
    int half;      // buckets per sign half (num_buckets/2 bidirectional, num_buckets otherwise)
    int exact;     // half/2: distances below this map to themselves
    int bidir;     // 1: j - i > 0 takes the upper half
    int nthr;      // half - 1 - exact
    int sat;       // first distance whose bucket is the clamp value (the table radius)
    int thr[kMaxT5Thresholds];
};

// Host: fills b from (num_buckets, max_distance, bidirectional); returns false on
// invalid parameters. Exact integer arithmetic.
bool t5_make_buckets(int num_buckets, int max_distance, int bidirectional, T5Buckets *b);

// Scalar bias per relative offset ("Relative position embeddings" page, sections "T5" and
// "Placement in the taxonomy"): T5 buckets of a [num_buckets, H] table, ALiBi -m_h |delta|
// from a [H] slope array, or a [H|1, 2R+1] table read at clip(delta, R) + R.
enum BiasKind : int { kBiasBuckets = 0, kBiasAlibi = 1, kBiasTable = 2 };

// Device status word (one per device), set by bounded waits that run out.
int *device_error_word();  // device address of the word for the current device, or null

// ---- fp32 SIMT path --------------------------------------------------------------------
struct SimtArgs {
    const float *q, *k, *v, *aK, *aV;
    long long ths;
    int clip_k, causal;
    float scale;
    const int *kv_len;
    const float *bias;  // scalar bias (see bias_kind) or null
    int bias_kind;      // BiasKind
    int bias_R;         // kBiasTable: the table's clip radius
    long long bias_hs;  // kBiasTable: elements between heads' rows (0 = one shared row)
    int B, H, n, d;
    float *out;
};
// t5 non-null: the scalar-bias variant (bias_kind says which bias; t5 is read for buckets)
cudaError_t launch_simt_f32(const SimtArgs &a, const T5Buckets *t5, cudaStream_t s);

// ---- label kernel ----------------------------------------------------------------------
cudaError_t launch_labels(int kind, int clip_k, const T5Buckets *t5, int n_q, int n_k,
                          int *labels, cudaStream_t s);

// ---- bf16 tcgen05 path -------------------------------------------------------------------
enum Mode : int { kShaw = 0, kT5 = 1 };

struct TcArgs {
    const void *q, *k, *v, *aK, *aV;
    long long ths;
    int clip_k, causal;
    float scale;
    const int *kv_len;
    const float *bias;  // kT5 mode: the scalar bias of bias_kind
    int bias_kind;      // BiasKind
    int bias_R;         // kBiasTable: the table's clip radius
    long long bias_hs;  // kBiasTable: elements between heads' rows (0 = one shared row)
    int B, H, n, d;
    void *out;
    int mode;           // kShaw, or kT5 for every scalar offset bias
    long long wait_limit;  // bound of every device wait in SM clock cycles (<= 0: 2e9)
    int withhold_q;        // test hook: withhold the first Q load of each producer (timeout test)
};
// Returns cudaErrorNotSupported for combinations the kernel does not cover (checked
// before any launch), cudaErrorInvalidValue for bad tensor-map parameters.
cudaError_t launch_tc_bf16_d64(const TcArgs &a, const T5Buckets *t5, int *err, cudaStream_t s);
cudaError_t launch_tc_bf16_d128(const TcArgs &a, const T5Buckets *t5, int *err, cudaStream_t s);
// Sequences of at most 256 keys with d = 64 and the Shaw tables (at most 64 staged rows):
// the short-sequence kernel. short_kernel_covers says whether it takes the call;
// launch_short_bf16 returns cudaErrorNotSupported for anything else (checked before any launch).
bool short_kernel_covers(const TcArgs &a);
cudaError_t launch_short_bf16(const TcArgs &a, int *err, cudaStream_t s);

// ---- bf16 decode step ----------------------------------------------------------------------
struct DecodeArgs {
    const void *q, *k_cache, *v_cache, *aK, *aV;
    long long ths;
    int clip_k;
    float scale;
    const int *cache_len;
    int B, H, T, d;
    void *out;
    void *workspace;  // device scratch for the split over all caches, or null
    unsigned long long workspace_bytes;
};
// bytes of workspace the split over all caches uses (0: more than 1024 sequences, or B * H * T
// beyond 2^50: one CTA per cache)
unsigned long long decode_workspace_bytes(int B, int H, int T, int d);
// cudaErrorNotSupported when clip_k + 1 table rows exceed the kernel's bins; without a large
// enough workspace the single-pass kernel runs
cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s);

// ---- gradients of the scalar offset biases (T5, ALiBi, per-offset table) ------------------
constexpr int kBiasBwdMaxN = 4096;  // the bias and the de sums of every offset sit in shared memory
struct BiasBwdArgs {
    const void *q, *k, *v, *dout;
    const float *bias;        // T5 [num_buckets, H], ALiBi slopes [H], table [H|1, 2R+1]
    int kind;                 // BiasKind
    int num_buckets;          // T5
    int radius;               // table
    long long head_stride;    // table: elements between heads' rows (0 = one shared row)
    int causal;
    float scale;
    const int *kv_len;
    int B, H, n, d;
    int bf16;
    float *dq, *dk, *dv, *dbias;
    void *workspace;
};
// floats of per-row records at the start of the workspace (G, the per-offset sums, follows)
long long bias_bwd_rec_floats(int B, int H, int n);
unsigned long long bias_bwd_workspace_bytes(int B, int H, int n);
// cudaErrorNotSupported for n > kBiasBwdMaxN or d > 128
cudaError_t launch_bias_bwd(const BiasBwdArgs &a, const T5Buckets *t5, cudaStream_t s);

// ---- labelled edges (SIMT, fp32 arithmetic) ----------------------------------------------
constexpr int kMaxLabels = 256;      // uint8 labels
constexpr int kLabelOutOfRange = 1;  // device status word value (RELATTN_ERR_INVALID_ARG)
struct LabeledArgs {
    const void *q, *k, *v, *aK, *aV;
    long long ths;            // elements between heads' tables (0 = shared)
    int num_labels;           // table rows
    const uint8_t *labels;    // [*, n, n]
    long long lbs;            // elements between sequences' label matrices (0 = shared)
    int causal;
    float scale;
    const int *kv_len;
    int B, H, n, d;
    int bf16;                 // 1: q, k, v, tables and out are bf16; 0: fp32
    void *out;
    int *err;                 // device status word (a label without a table row)
    long long wait_limit;     // tensor-core path: bound of every device wait (cycles, <= 0: 2e9)
};
// SIMT kernel; cudaErrorNotSupported when d > 128 or more than 256 labels
cudaError_t launch_labeled(const LabeledArgs &a, cudaStream_t s);
// tensor-core kernel (bf16, d = 64 or 128, at most 128 labels); cudaErrorNotSupported for any
// other combination, checked before any launch
cudaError_t launch_labeled_tc(const LabeledArgs &a, cudaStream_t s);

// ---- Transformer-XL relative attention (SIMT, fp32 arithmetic) -----------------------------
struct TxlArgs {
    const void *q, *k, *v;   // [B, H, n, d]
    const void *rel;         // [H|1, 2n - 1, d]: the projected encoding of offset j - i at row j - i + n - 1
    const void *u, *vb;      // [H|1, d]: the global content and position biases
    int shared;              // 1: rel, u and vb are one set for every head
    int causal;
    float scale;
    const int *kv_len;
    int B, H, n, d;
    int bf16;
    void *out;
    int *err;               // tensor-core path: device status word
    long long wait_limit;   // tensor-core path: bound of every device wait (cycles, <= 0: 2e9)
};
// SIMT kernel; cudaErrorNotSupported when d > 128
cudaError_t launch_txl(const TxlArgs &a, cudaStream_t s);
// the sinusoidal encodings of the offsets -(n-1) .. n-1: [2n - 1, d_model] of bf16 or fp32
cudaError_t launch_sinusoid(int n, int d_model, int bf16, void *out, cudaStream_t s);
// tensor-core kernel (bf16, d = 64 or 128); txl_tc_covers says whether it takes the call
bool txl_tc_covers(const TxlArgs &a);
cudaError_t launch_txl_tc(const TxlArgs &a, cudaStream_t s);

// ---- gradients (SIMT, fp32 arithmetic) ---------------------------------------------------
struct BwdArgs {
    const void *q, *k, *v, *aK, *aV, *dout;
    long long ths;
    int clip_k, causal;
    float scale;
    const int *kv_len;
    int B, H, n, d;
    int bf16;  // 1: q, k, v, tables and dout are bf16; 0: fp32
    float *dq, *dk, *dv, *daK, *daV;
    void *workspace;  // at least bwd_workspace_bytes
    int *err;               // device status word (tensor-core waits; out-of-range labels)
    long long wait_limit;   // tensor-core path: bound of every device wait (cycles, <= 0: 2e9)
    // labelled edges (SIMT only): the table row of pair (i, j) is labels[b * lbs + i * n + j]
    // (num_labels rows) in place of clip(j - i, clip_k) + clip_k
    const uint8_t *labels;
    long long lbs;
    int num_labels;
};
// the larger of the two paths' needs
unsigned long long bwd_workspace_bytes(int B, int H, int n, int clip_k);
// the SIMT kernels' need for W table rows (2k+1, or the number of labels)
unsigned long long bwd_simt_workspace_bytes(int B, int H, int n, int W);
// SIMT kernels; cudaErrorNotSupported when the table rows exceed 257 or d > 128
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t s);
// tensor-core kernels (bf16, d = 64 or 128, at most 128 staged table rows, workspace aligned
// to 256 bytes); bwd_tc_covers says whether they take the call
unsigned long long bwd_tc_workspace_bytes(int B, int H, int n, int clip_k);
bool bwd_tc_covers(const BwdArgs &a);
cudaError_t launch_bwd_tc(const BwdArgs &a, cudaStream_t s);

}  // namespace relattn
