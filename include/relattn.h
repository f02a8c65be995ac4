/*
 * relattn — relation-aware self-attention forward for GB300 (sm_103a), C ABI.
 *
 * Method: Shaw, Uszkoreit & Vaswani, "Self-Attention with Relative Position
 * Representations" (paper summary page, section 3.4: eq. 3 for the output, eq. 4 for the
 * compatibility, clip(j - i, k) and the 2k+1 edge vectors w_{-k}..w_{k}; section
 * "Efficient Implementation" for the eq. 5 split). T5 variant: "Relative position
 * embeddings" page, section "T5"; ALiBi and the per-offset scalar table: the same page,
 * sections "Placement in the taxonomy" and "Two-dimensional variants". Labelled edges: the
 * section "Relation-Aware Self-Attention: The Core Modification" of the same page. Also a
 * decode step against a key/value cache, the gradients of relattn_fwd, of the labelled-edge
 * forward and of the scalar offset biases.
 *
 * Conventions shared by every entry point
 *   - Tensors q, k, v, out are [B, H, n, d], contiguous, d fastest (row-major).
 *   - Every tensor pointer is caller-owned DEVICE memory, 16-byte aligned. The library
 *     never allocates, frees or keeps a pointer after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Nothing is synchronised; there is no CPU fallback.
 *   - Arguments are validated on the host before any launch: a bad argument returns
 *     RELATTN_ERR_INVALID_ARG, a valid but unimplemented combination returns
 *     RELATTN_ERR_UNSUPPORTED, and a failed launch returns RELATTN_ERR_CUDA. In all three
 *     cases nothing was enqueued.
 *   - Device-side waits are bounded (about one second); a wait that runs out records
 *     RELATTN_ERR_TIMEOUT in a device status word, which relattn_get_device_error reads.
 */
#ifndef RELATTN_H
#define RELATTN_H

#if defined(__GNUC__)
#define RELATTN_API __attribute__((visibility("default")))
#else
#define RELATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RELATTN_OK = 0,
    RELATTN_ERR_INVALID_ARG = 1,
    RELATTN_ERR_UNSUPPORTED = 2,
    RELATTN_ERR_CUDA = 3,
    RELATTN_ERR_TIMEOUT = 4
} relattn_status_t;

/* Element type of q, k, v, the Shaw tables and out. */
typedef enum {
    RELATTN_BF16 = 0, /* tcgen05 tensor-core path: d in {64, 128} */
    RELATTN_F32 = 1   /* fp32 SIMT path: 1 <= d <= 128 */
} relattn_dtype_t;

struct CUstream_st;
typedef struct CUstream_st *relattn_stream_t; /* same type as cudaStream_t */

/*
 * relattn_fwd — Shaw relation-aware self-attention forward (eq. 3 and eq. 4).
 *
 *   e_ij = scale * q_i . (k_j + aK[h][clip(j - i, clip_k) + clip_k])
 *   z_i  = sum_j softmax_j(e)_ij * (v_j + aV[h][clip(j - i, clip_k) + clip_k])
 *
 * over the allowed keys j: j < kv_len[b] (all j when kv_len is NULL) and, if causal,
 * j <= i. A row with no allowed key is written as zeros.
 *
 *   q, k, v           [B, H, n, d] of `dtype`.
 *   aK, aV            edge tables [*, 2*clip_k + 1, d] of `dtype`, row r holding
 *                     w_{r - clip_k} (row 0 = w_{-k}). NULL drops that term (aV NULL is
 *                     the key-only mode; both NULL is plain attention).
 *   table_head_stride elements between consecutive heads' tables; 0 = one table shared
 *                     by all heads. Otherwise >= (2*clip_k + 1) * d and, for bf16, a
 *                     multiple of 8.
 *   clip_k            clipping distance k >= 0.
 *   causal            0 or 1.
 *   scale             multiplies the whole compatibility (content and edge terms);
 *                     1/sqrt(d) in the paper.
 *   kv_len            [B] int32 device array of key lengths, or NULL.
 *   out               [B, H, n, d] of `dtype`; must not alias an input.
 *
 * bf16 limits (else RELATTN_ERR_UNSUPPORTED): the staged table rows (clip_k + 1 when
 * causal, else 2*clip_k + 1) must be <= 128.
 */
RELATTN_API relattn_status_t relattn_fwd(const void *q, const void *k, const void *v,
                             const void *aK, const void *aV, long long table_head_stride,
                             int clip_k, int causal, float scale, const int *kv_len,
                             int B, int H, int n, int d, int dtype,
                             void *out, relattn_stream_t stream);

/*
 * relattn_t5bias_fwd — T5 scalar bucketed relative bias ("Relative position embeddings",
 * section "T5"):
 *
 *   e_ij = scale * q_i . k_j + bias[bucket(j - i) * H + h]
 *
 * softmax and output as above (no edge vector on the values). bias is a [num_buckets, H]
 * fp32 device array. bucket(): bidirectional splits the buckets into two halves of
 * num_buckets/2, one per sign (j - i > 0 takes the upper half), each exact below
 * half/2 and logarithmic up to max_distance, clamped to the half's last bucket;
 * unidirectional uses one half of num_buckets on max(i - j, 0). The floor in the
 * logarithmic part is exact (integer arithmetic on the host). T5 itself uses scale = 1.
 *
 * Requires 4 <= num_buckets <= 256 (bidirectional) or 2 <= num_buckets <= 256, and
 * max_distance greater than the exact range, else RELATTN_ERR_INVALID_ARG.
 */
RELATTN_API relattn_status_t relattn_t5bias_fwd(const void *q, const void *k, const void *v,
                                    const float *bias, int num_buckets, int max_distance,
                                    int bidirectional, int causal, float scale,
                                    const int *kv_len, int B, int H, int n, int d, int dtype,
                                    void *out, relattn_stream_t stream);

/*
 * relattn_alibi_fwd — ALiBi: the scalar relative bias with the T5 table replaced by a
 * fixed line per head ("Relative position embeddings", section "Placement in the taxonomy"):
 *
 *   e_ij = scale * q_i . k_j - slopes[h] * |j - i|
 *
 * softmax, masks, empty rows and output as in relattn_fwd (no edge vector on the values).
 * slopes is a [H] fp32 device array (the method fixes them, e.g. 2^(-8(h+1)/H); any values
 * are accepted). The bias is formed in fp32 (slope times the exact distance).
 *
 * bf16 limit (else RELATTN_ERR_UNSUPPORTED): the kernel holds the bias of every offset of
 * the sequence in shared memory, 4 * (2n + 127) bytes per query tile in flight; n up to
 * about 20000 fits. fp32 (SIMT) has no such limit.
 */
RELATTN_API relattn_status_t relattn_alibi_fwd(const void *q, const void *k, const void *v,
                                   const float *slopes, int causal, float scale,
                                   const int *kv_len, int B, int H, int n, int d, int dtype,
                                   void *out, relattn_stream_t stream);

/*
 * relattn_offset_bias_fwd — a learned scalar per relative offset, clipped like the Shaw
 * tables: the T5 form ("Relative position embeddings", section "T5") with one table entry
 * per offset instead of per bucket (the 1-D case of the offset-indexed table of section
 * "Two-dimensional variants"), read at clip(j - i, radius):
 *
 *   e_ij = scale * q_i . k_j + table[h * table_head_stride + clip(j - i, radius) + radius]
 *
 * softmax, masks, empty rows and output as in relattn_fwd. table is an fp32 device array
 * [H|1, 2*radius + 1], entry r holding the bias of offset r - radius.
 *   table_head_stride  elements between heads' rows; 0 = one row shared by every head,
 *                      else >= 2*radius + 1.
 *   radius             0 <= radius <= 2^20 (radius >= n - 1 means no clipping).
 * bf16 limit (else RELATTN_ERR_UNSUPPORTED): as relattn_alibi_fwd, with min(radius, n - 1)
 * in place of n - 1.
 */
RELATTN_API relattn_status_t relattn_offset_bias_fwd(const void *q, const void *k, const void *v,
                                   const float *table, long long table_head_stride, int radius,
                                   int causal, float scale, const int *kv_len, int B, int H,
                                   int n, int d, int dtype, void *out, relattn_stream_t stream);

/*
 * relattn_labeled_fwd — relation-aware attention over arbitrary labelled edges (paper
 * summary page, section "Relation-Aware Self-Attention: The Core Modification": every edge
 * (i, j) of the input graph carries its own a^K_ij and a^V_ij; section 3.4 specialises the
 * label to clip(j - i, k) + k, which relattn_fwd computes without a label matrix):
 *
 *   e_ij = scale * q_i . (k_j + aK[h][L])
 *   z_i  = sum_j softmax_j(e)_ij * (v_j + aV[h][L]),     L = labels[b * label_batch_stride + i * n + j]
 *
 * masks, empty rows and output as in relattn_fwd.
 *   aK, aV              tables [*, num_labels, d] of `dtype` (16-byte aligned); NULL drops
 *                       that term (both NULL: plain attention, labels unused and may be NULL).
 *   table_head_stride   elements between heads' tables; 0 = shared; else >= num_labels * d
 *                       and a multiple of 8 (bf16) / 4 (fp32).
 *   num_labels          1 .. 256.
 *   labels              uint8 device array of labels, [B|1, n, n] row-major.
 *   label_batch_stride  elements between sequences' label matrices; 0 = one matrix for
 *                       every sequence, else >= n * n.
 * A label >= num_labels is not checked on the host: the kernel reads it as the last table
 * row and sets the device status word to RELATTN_ERR_INVALID_ARG (relattn_get_device_error).
 * bf16 with d = 64 or 128 and at most 128 labels (when the tables' rows fit shared memory)
 * runs on the tensor cores: R = Q aK^T over the labels per query tile, gathered by label into
 * the scores, and per-label bins of the probabilities times aV, fp32 accumulation. Every other
 * supported shape runs on the SIMT units with fp32 arithmetic; d <= 128 and a multiple of
 * 8 (bf16) / 4 (fp32), else RELATTN_ERR_UNSUPPORTED.
 */
RELATTN_API relattn_status_t relattn_labeled_fwd(const void *q, const void *k, const void *v,
                                     const void *aK, const void *aV, long long table_head_stride,
                                     int num_labels, const unsigned char *labels,
                                     long long label_batch_stride, int causal, float scale,
                                     const int *kv_len, int B, int H, int n, int d, int dtype,
                                     void *out, relattn_stream_t stream);

/*
 * relattn_txl_fwd — Transformer-XL relative attention ("Relative Position Encoding in
 * Transformer-XL" page: the four-term score and the roles of the global biases u and v;
 * "Relative position embeddings" page, section "Transformer-XL"):
 *
 *   A_ij = q_i . k_j + q_i . r_ij + u . k_j + v . r_ij,    r_ij = rel[h][j - i + n - 1]
 *   z_i  = sum_j softmax_j(scale * A)_ij v_j
 *
 * over the allowed keys (j < kv_len[b], and j <= i if causal); a row with no allowed key is
 * written as zeros. Unlike relattn_fwd the offsets are not clipped and there is no value term.
 *   q, k, v           [B, H, n, d] of `dtype` (16-byte aligned).
 *   rel               [H, 2n - 1, d] of `dtype` (16-byte aligned): row o holds the projected
 *                     encoding of the offset j - i = o - (n - 1), i.e. W_{k,R} r(j - i).
 *   u, vb             [H, d] of `dtype`: the global content bias u and position bias v.
 *   shared            1: rel, u and vb are a single set ([1, 2n - 1, d], [1, d]) for all heads.
 *   causal, scale, kv_len, B, H, n, d, dtype, out, stream   as in relattn_fwd; d <= 128 and a
 *                     multiple of 8 (bf16) / 4 (fp32), else RELATTN_ERR_UNSUPPORTED.
 * bf16 with d = 64 or 128 runs on the tensor cores: per (query tile, key tile) S = Q K^T and
 * T = Q R^T over the 255 offsets the pair spans (R: the table rows of those offsets), T read
 * along its diagonals, u . k_j and v . r_ij added as per-key and per-offset fp32 scalars,
 * O += P V with P in bf16, fp32 accumulation. Everything else (fp32, other d) runs on the SIMT
 * units with fp32 arithmetic: one warp per query row, the two dot products (q_i + u) . k_j and
 * (q_i + v) . r_ij per key. Device waits of the tensor-core path are bounded as in relattn_fwd.
 */
RELATTN_API relattn_status_t relattn_txl_fwd(const void *q, const void *k, const void *v,
                                 const void *rel, const void *u, const void *vb, int shared,
                                 int causal, float scale, const int *kv_len, int B, int H, int n,
                                 int d, int dtype, void *out, relattn_stream_t stream);

/*
 * relattn_decode_fwd — one incremental decoding step of a causal decoder: the new token of
 * every sequence attends to its sequence's key/value cache with the relative terms of
 * relattn_fwd ("Self-Attention with Relative Position Representations" page, section 3.4, eq. 3 and eq. 4 with clip(j - i, k)).
 * With t = cache_len[b] - 1, the new token's position (its own key and value are already
 * the cache's row t):
 *
 *   e_j = scale * q . (k_j + aK[h][clip(j - t, clip_k) + clip_k]),   j = 0 .. t
 *   z   = sum_j softmax_j(e)_j * (v_j + aV[h][clip(j - t, clip_k) + clip_k])
 *
 * i.e. row t of relattn_fwd with causal = 1 over the sequence's first t + 1 positions.
 * Only table rows 0 .. clip_k (offsets -k .. 0) are read.
 *
 *   q                 [B, H, d] bf16: the new tokens' queries.
 *   k_cache, v_cache  [B, H, T, d] bf16 caches of capacity T; rows >= cache_len[b] are
 *                     not read.
 *   aK, aV, table_head_stride, clip_k, scale   as in relattn_fwd (bf16 tables).
 *   cache_len         [B] int32 device array, each in 0 .. T (larger values are taken as
 *                     T); a sequence with cache_len 0 gets zeros.
 *   out               [B, H, d] bf16; must not alias an input.
 *
 *   workspace         caller-owned device scratch of workspace_bytes (16-byte aligned),
 *                     or NULL. When relattn_decode_workspace_size is not 0 (at most 1024
 *                     sequences) and the workspace is that large, the cached keys of all
 *                     sequence-heads are cut into equal ranges, one per CTA of a grid that
 *                     fills the GPU once, whatever the mix of cache lengths; a second kernel
 *                     on the same stream merges the ranges of each cache and adds the value
 *                     bins. Otherwise one CTA reads a whole cache. The contents are scratch
 *                     on entry and on return, and two calls running at the same time must
 *                     not share it.
 *
 * bf16 only, d in {64, 128}; clip_k <= 256 (else RELATTN_ERR_UNSUPPORTED). Appending the
 * new token's key and value to the cache is the caller's job.
 */
RELATTN_API relattn_status_t relattn_decode_fwd(const void *q, const void *k_cache,
                                    const void *v_cache, const void *aK, const void *aV,
                                    long long table_head_stride, int clip_k, float scale,
                                    const int *cache_len, int B, int H, int T, int d,
                                    void *workspace, unsigned long long workspace_bytes,
                                    void *out, relattn_stream_t stream);

/*
 * relattn_decode_fwd_noalloc — relattn_decode_fwd for callers that cannot allocate device
 * memory: a host runtime that reserves its whole device budget at start-up and forbids
 * allocations afterwards, or a plugin inside another engine that is handed tensors but no
 * allocator. cudaMalloc may also synchronise the device, which a latency-bound decoding loop
 * cannot afford. The arguments are those of relattn_decode_fwd without workspace /
 * workspace_bytes; the scratch is a 4 MiB array that is part of the library's device image
 * (a file-scope __device__ array, held by every device that loads the library until the
 * process exits), so no call allocates anything.
 *
 *   - When the split would need more than 4 MiB (relattn_decode_workspace_size > 4 MiB:
 *     more than about 7000 sequence-heads at d = 128, 13000 at d = 64), the call runs
 *     without the split, one CTA per cache, and uses no scratch.
 *   - The array is one per device and shared by every call of this entry point on that
 *     device: calls that overlap on the GPU (different streams, no ordering) race on it and
 *     give wrong results; calls on one stream are ordered. Each call writes every scratch
 *     value it later reads, so nothing has to be cleared between calls.
 *   - The first call on a device, with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress) and keeps it for the process; make that first call
 *     before any stream capture. The kept address is not valid after cudaDeviceReset: do not
 *     use the library across a reset.
 *
 * The pages describe no counterpart of this entry point: it is an interface convenience,
 * not part of the method.
 */
RELATTN_API relattn_status_t relattn_decode_fwd_noalloc(const void *q, const void *k_cache,
                                            const void *v_cache, const void *aK,
                                            const void *aV, long long table_head_stride,
                                            int clip_k, float scale, const int *cache_len,
                                            int B, int H, int T, int d, void *out,
                                            relattn_stream_t stream);

/*
 * relattn_decode_workspace_size — host only: the workspace bytes relattn_decode_fwd uses
 * to split the caches over the GPU: a length prefix over the sequences and one
 * {maximum, row sum, P V[d]} record per (CTA, sequence-head) segment, (1024 + B H) records
 * at most; 0 when it runs one CTA per cache (more than 1024 sequences, or B H T > 2^50).
 */
RELATTN_API relattn_status_t relattn_decode_workspace_size(int B, int H, int T, int d,
                                               unsigned long long *bytes);

/*
 * relattn_sinusoid_table — the fixed sinusoidal encodings of every relative offset of a
 * length-n sequence, the r of the Transformer-XL score before its projection ("Relative
 * Position Encoding in Transformer-XL" page: r_{i-j} is a sinusoid of the distance, in the
 * form the "Self-Attention with Relative Position Representations" page states for the
 * original Transformer's position encodings):
 *
 *   out[o][2i]     = sin(p / 10000^(2i / d_model)),
 *   out[o][2i + 1] = cos(p / 10000^(2i / d_model)),     p = o - (n - 1),  o = 0 .. 2n - 2.
 *
 * The angle is formed in fp64, the values rounded to `dtype` (RELATTN_BF16 or RELATTN_F32).
 * out: caller-owned device memory of (2n - 1) * d_model elements; d_model even and >= 2.
 * Projected by the head's W_{k,R} (a plain matrix product, [H, d, d_model] times this table)
 * it gives the `rel` argument of relattn_txl_fwd.
 */
RELATTN_API relattn_status_t relattn_sinusoid_table(int n, int d_model, int dtype, void *out,
                                        relattn_stream_t stream);

/*
 * relattn_bwd — gradients of relattn_fwd (Shaw relation-aware attention) for training. The
 * pages state only the forward pass ("Self-Attention with Relative Position Representations" page, section 3.4, eq. 3 and eq. 4);
 * these are the chain rule through it:
 *
 *   dp_ij = dz_i . (v_j + aV_r),  de_ij = p_ij (dp_ij - sum_j' p_ij' dp_ij'),
 *   dq_i = scale sum_j de_ij (k_j + aK_r),  dk_j = scale sum_i de_ij q_i,
 *   dv_j = sum_i p_ij dz_i,  daK_r = scale sum_{r_ij = r} de_ij q_i,
 *   daV_r = sum_{r_ij = r} p_ij dz_i,     r = r_ij = clip(j - i, clip_k) + clip_k,
 *
 * with p the forward's softmax over the same allowed keys (causal, kv_len).
 *
 *   q, k, v, aK, aV, table_head_stride, clip_k, causal, scale, kv_len, B, H, n, d, dtype
 *                     as in relattn_fwd (bf16 or fp32; any 1 <= d <= 128).
 *   dout              [B, H, n, d] of `dtype`: the gradient of the loss with respect to out.
 *   dq, dk, dv        [B, H, n, d] fp32, written (not accumulated).
 *   daK, daV          fp32 tables laid out like aK / aV (head stride table_head_stride;
 *                     with 0 one table receives every head's gradient); written (not
 *                     accumulated); required when the matching table is given, ignored
 *                     otherwise.
 *   workspace         caller-owned device scratch of at least relattn_bwd_workspace_size
 *                     bytes (4-byte aligned; 256-byte aligned for the tensor-core path);
 *                     its contents are scratch (per query row: the softmax statistics, the
 *                     relative terms R and Rv with them folded in, the bins).
 *
 * Two paths (relattn_set_bwd_tensor_cores chooses). Tensor cores, for bf16 with d = 64 or
 * 128 and at most 128 staged table rows (clip_k + 1 causal, 2*clip_k + 1 otherwise): a
 * query-tile kernel forms S = Q K^T and dP = dZ V^T on tcgen05 and takes each row's softmax
 * statistics and bins; a key-tile kernel recomputes S^T and dP^T, forms P and dS and
 * accumulates dV = P^T dZ and dK = dS^T Q in tensor memory, adding dQ = dS K into dq with
 * atomic adds; a SIMT kernel adds the table terms of dq and the table gradients. P, dS and
 * the bins enter the products as bf16 (fp32 accumulation). SIMT, for everything else
 * (fp32 inputs, any 1 <= d <= 128, 2*clip_k + 1 <= 257): fp32 arithmetic from the exact
 * inputs, three kernels (one warp per query row, one warp per key, one CTA per table row).
 * Device waits of the tensor-core path are bounded as in relattn_fwd (relattn_set_wait_limit;
 * RELATTN_ERR_TIMEOUT through relattn_get_device_error).
 */
RELATTN_API relattn_status_t relattn_bwd(const void *q, const void *k, const void *v,
                             const void *aK, const void *aV, long long table_head_stride,
                             int clip_k, int causal, float scale, const int *kv_len, int B,
                             int H, int n, int d, int dtype, const void *dout, float *dq,
                             float *dk, float *dv, float *daK, float *daV, void *workspace,
                             unsigned long long workspace_bytes, relattn_stream_t stream);

/* relattn_bwd_workspace_size — host only: the workspace bytes relattn_bwd needs. */
RELATTN_API relattn_status_t relattn_bwd_workspace_size(int B, int H, int n, int d, int clip_k,
                                            unsigned long long *bytes);

/*
 * relattn_scalar_bias_bwd — gradients of the scalar offset-bias forwards: relattn_t5bias_fwd
 * (kind 0, "Relative position embeddings" page, section "T5"), relattn_alibi_fwd (kind 1,
 * same page, "Placement in the taxonomy": -m_h |j - i|) and relattn_offset_bias_fwd (kind 2,
 * a learned scalar per offset clipped at `radius`). The pages give only the forward; these
 * are the chain rule through e_ij = scale q_i . k_j + b_h(j - i) and the softmax:
 *
 *   dq_i = scale sum_j de_ij k_j,   dk_j = scale sum_i de_ij q_i,   dv_j = sum_i p_ij dz_i,
 *   de_ij = p_ij (dz_i . v_j - D_i),   D_i = sum_j p_ij dz_i . v_j,
 *
 * and the parameter's gradient from the per-offset sums G_h(o) = sum_(b,i) de_(i,i+o):
 *   kind 0: bias [num_buckets, H] fp32 -> dbias [num_buckets, H], dbias[c, h] = sum of
 *           G_h(o) over the offsets o of bucket c (num_buckets, max_distance, bidirectional as
 *           in relattn_t5bias_fwd);
 *   kind 1: slopes [H] fp32 -> dbias [H] = -sum_o |o| G_h(o);
 *   kind 2: table rows of 2*radius + 1 fp32 at bias_head_stride elements between heads (0: one
 *           shared row) -> dbias of the same layout, dbias[h, r] = sum of G_h(o) over the
 *           offsets with clip(o, radius) + radius = r (a shared row sums over the heads);
 *           every entry of the rows is written.
 *
 *   q, k, v, dout, causal, scale, kv_len, B, H, n, d, dtype   as in the forward (bf16 or
 *                     fp32 inputs, d <= 128, n <= 4096, B * H <= 65535; else
 *                     RELATTN_ERR_UNSUPPORTED).
 *   dq, dk, dv        [B, H, n, d] fp32; padded keys get zero; rows with no allowed key zero.
 *   workspace         caller-owned device scratch of at least
 *                     relattn_scalar_bias_bwd_workspace_size bytes (4-byte aligned): per row
 *                     the softmax statistics, then G. Contents are scratch.
 *
 * fp32 arithmetic on the SIMT units (the bias term has no contraction of its own); every
 * output is written (nothing needs clearing). Arguments that fail a check return
 * RELATTN_ERR_INVALID_ARG before any launch.
 */
RELATTN_API relattn_status_t relattn_scalar_bias_bwd(const void *q, const void *k, const void *v,
                                         const void *dout, int kind, const float *bias,
                                         int num_buckets, int max_distance, int bidirectional,
                                         int radius, long long bias_head_stride, int causal,
                                         float scale, const int *kv_len, int B, int H, int n,
                                         int d, int dtype, float *dq, float *dk, float *dv,
                                         float *dbias, void *workspace,
                                         unsigned long long workspace_bytes,
                                         relattn_stream_t stream);

/* relattn_scalar_bias_bwd_workspace_size — host only: the workspace bytes it needs. */
RELATTN_API relattn_status_t relattn_scalar_bias_bwd_workspace_size(int B, int H, int n,
                                                        unsigned long long *bytes);

/*
 * relattn_labeled_bwd — gradients of relattn_labeled_fwd (the labelled-edge forward; paper
 * summary page, section "Relation-Aware Self-Attention: The Core Modification"): relattn_bwd's
 * chain rule with the table row of pair (i, j) read from the label matrix,
 * r_ij = labels[b * label_batch_stride + i * n + j], in place of clip(j - i, k) + k:
 *
 *   dq_i = scale sum_j de_ij (k_j + aK[h][r_ij]),  dk_j = scale sum_i de_ij q_i,
 *   dv_j = sum_i p_ij dz_i,  daK[h][r] = scale sum_{r_ij = r} de_ij q_i,
 *   daV[h][r] = sum_{r_ij = r} p_ij dz_i,   de_ij = p_ij (dz_i . (v_j + aV[h][r_ij]) - D_i).
 *
 *   arguments as in relattn_labeled_fwd (num_labels 1 .. 256, labels required) and relattn_bwd
 *   (dout of q's dtype; dq, dk, dv [B, H, n, d] fp32; daK / daV fp32 of the tables' layout,
 *   required with their table and written whole; d <= 128).
 *   workspace         caller-owned device scratch of at least relattn_labeled_bwd_workspace_size
 *                     bytes (4-byte aligned); its contents are scratch.
 * A label >= num_labels is read as the last table row and sets the device status word to
 * RELATTN_ERR_INVALID_ARG, as in the forward. fp32 arithmetic on the SIMT units.
 */
RELATTN_API relattn_status_t relattn_labeled_bwd(const void *q, const void *k, const void *v,
                                     const void *aK, const void *aV, long long table_head_stride,
                                     int num_labels, const unsigned char *labels,
                                     long long label_batch_stride, int causal, float scale,
                                     const int *kv_len, int B, int H, int n, int d, int dtype,
                                     const void *dout, float *dq, float *dk, float *dv,
                                     float *daK, float *daV, void *workspace,
                                     unsigned long long workspace_bytes, relattn_stream_t stream);

/* relattn_labeled_bwd_workspace_size — host only: the workspace bytes it needs. */
RELATTN_API relattn_status_t relattn_labeled_bwd_workspace_size(int B, int H, int n,
                                                    int num_labels,
                                                    unsigned long long *bytes);

/*
 * relattn_labels — the integer edge label of every (i, j), computed by the same device
 * functions the attention kernels use, written as int32 labels[i * n_k + j].
 *   kind 0: clip row clip(j - i, clip_k) + clip_k ("Self-Attention with Relative Position Representations" page, section 3.4).
 *   kind 1: T5 bucket(j - i) with (num_buckets, max_distance, bidirectional).
 * labels is caller-owned device memory of n_q * n_k int32.
 */
RELATTN_API relattn_status_t relattn_labels(int kind, int clip_k, int num_buckets, int max_distance,
                                int bidirectional, int n_q, int n_k, int *labels,
                                relattn_stream_t stream);

/*
 * relattn_t5_thresholds — host only, no GPU needed. Writes the exact first distance a of
 * each logarithmic T5 bucket (buckets exact+1 .. half-1 of one half) into
 * thresholds[0 .. *count - 1]; capacity is the array length.
 */
RELATTN_API relattn_status_t relattn_t5_thresholds(int num_buckets, int max_distance, int bidirectional,
                                       int *thresholds, int capacity, int *count);

/*
 * relattn_get_device_error — synchronises `stream`, then reads and clears the device
 * status word of the current device: RELATTN_OK, RELATTN_ERR_TIMEOUT if a bounded
 * device wait ran out since the last call, or RELATTN_ERR_INVALID_ARG if relattn_labeled_fwd
 * met a label without a table row. RELATTN_ERR_CUDA if the stream reports an error.
 */
RELATTN_API relattn_status_t relattn_get_device_error(relattn_stream_t stream);

/*
 * relattn_set_wait_limit — the bound of every device-side wait of the tensor-core forward
 * kernels (relattn_fwd, relattn_t5bias_fwd, relattn_alibi_fwd, relattn_offset_bias_fwd on
 * bf16), in SM clock cycles; the default is 2e9 (about one second at 2 GHz). A wait that
 * runs out makes every warp of the kernel stop, wait (again bounded) for its copies and
 * tensor-core operations in flight, release its tensor memory and exit; the call's output is
 * then undefined and relattn_get_device_error reports RELATTN_ERR_TIMEOUT. The setting is
 * process-wide and applies to launches made after the call. 1000 <= cycles <= 2^40, else
 * RELATTN_ERR_INVALID_ARG. Host only; not part of the method (the pages have no
 * counterpart): failure detection of the library.
 */
RELATTN_API relattn_status_t relattn_set_wait_limit(long long cycles);

/*
 * relattn_debug_withhold_first_load — test hook for the timeout path: with on = 1, each
 * producer warp of the tensor-core forward kernels announces the Q tiles of its first work
 * item to their barrier but never loads them, so the tensor-core warp's bounded wait for
 * them runs out (no fault, no trap: the kernel exits through its abort path). on = 0
 * (the default) restores normal launches. Process-wide; never set it in production.
 */
RELATTN_API relattn_status_t relattn_debug_withhold_first_load(int on);

/*
 * relattn_set_short_kernel — routing switch of the bf16 forward. With on = 1 (the default),
 * relattn_fwd calls with n <= 256, d = 64 and at most 64 staged table rows (clip_k + 1
 * causal, 2*clip_k + 1 otherwise) run on the short-sequence kernel, which keeps all of a
 * query tile's keys on chip and runs two CTAs per SM; on = 0 sends them to the general
 * kernel. Both compute the same eq. 3 / eq. 4 (results agree to rounding). Process-wide,
 * read at each call; any other value is RELATTN_ERR_INVALID_ARG.
 */
RELATTN_API relattn_status_t relattn_set_short_kernel(int on);

/*
 * relattn_set_bwd_tensor_cores — routing switch of relattn_bwd. With on = 1 (the default),
 * bf16 calls with d = 64 or 128, at most 128 staged table rows (clip_k + 1 causal,
 * 2*clip_k + 1 otherwise) and a workspace aligned to 256 bytes run on the tensor-core
 * kernels; on = 0 sends them to the SIMT kernels (fp32 arithmetic from the exact inputs).
 * Both compute the same gradients, the tensor-core path with bf16 operands in its products
 * (P, dS and the bins rounded to bf16). Process-wide, read at each call; any other value
 * is RELATTN_ERR_INVALID_ARG.
 */
RELATTN_API relattn_status_t relattn_set_bwd_tensor_cores(int on);

/* Static English text for a status code. */
RELATTN_API const char *relattn_status_string(relattn_status_t s);

/* Library version as 10000*major + 100*minor + patch. */
RELATTN_API int relattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RELATTN_H */
