/*
 * kvb.h -- C ABI of libkvb, closed-form cross-model KV-cache transfer on GB300.
 *
 * The method (Heo et al., "Cross-Model KV Cache Transfer in LLM Families"),
 * as the pages state it:
 *   "Cross-Model KV Transfer -- Reuse One Model's Prefill in Another"
 *   (VeloxQuant-MLX docs), section "The mapping":
 *       K_hat_t = rope_t( strip_rope_s(K_s)[sel] . W_K + b_K )
 *       V_hat_t =               V_s[sel]    . W_V + b_V
 *   "KVBridge" README, section "Loading":
 *       W = (X^T X + lambda I)^-1 X^T Y,  b = Ybar - Xbar W  on centered data,
 *       batchwise Chan/Welford merges of the centered statistics;
 *   "KVBridge" README, table "What ships": head-averaged single-source R^2,
 *       then top-k cross-layer, cross-head features.
 *
 * Layouts (all row-major, innermost last):
 *   cache      [L][H][T][d]   (layer, kv head, token, dim) -- "Before Mapping KV
 *                             Caches, Make Them Measurable", "what became
 *                             first-class".  Ragged batches pack sequences on T
 *                             with positions restarting at 0 per sequence.
 *   features   X_t[token][(j*H + h)*d + e] = cache[sel[t][j]][h][token][e]
 *                             (selected layers in the order given, then head,
 *                             then dim); p = k*H*d columns.
 *   W          [L_tgt][q][p], q = H*d: row n holds the p input weights of
 *                             output column n (a linear layer's weight layout;
 *                             the mathematical W is its transpose).
 *   bias       [L_tgt][q] float32.
 *   sel        [L_tgt][k] int32 on the HOST, one table for K and one for V.
 *   positions  [T] int32 on the DEVICE, 0 <= pos < max_pos (checked in the
 *                             kernels; a bad position sets KVB_ERR_INVALID_ARG
 *                             on the context and its rows are written as 0).
 *
 * RoPE: rotate-half pairs (i, i + d/2), frequency theta^(-2i/d); angles are
 * reduced in float64 once per context into float32 cos/sin tables.
 *
 * Ownership: the caller owns every tensor passed in.  The library allocates
 * only inside a context (RoPE tables, strip scratch, error word) and a
 * statistics object, and frees on destroy.
 *
 * Streams and errors: calls enqueue work on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and return without a host sync, except
 * kvb_layer_select, which syncs `stream` to hand back the selection.
 * Arguments are validated on the host before any launch.  No call aborts the
 * process: every failure is a returned status, with a message from
 * kvb_last_error().  Errors found by the kernels themselves (a bad position,
 * a bounded device wait that gave up) are recorded on the context and returned
 * by kvb_ctx_check() and by the next call on that context.
 *
 * Environment: KVB_WAIT_TIMEOUT_MS (default 2000) bounds every device-side
 * wait, read when a context is created (kvb_map_apply_noalloc, which has no
 * context, reads it on every call).  KVB_FIT_WORKSPACE_MB, read on every
 * call, caps the solver workspace of kvb_layer_select and kvb_ridge_solve
 * (default: half the free device memory, between 4 and 48 GiB); under a lower
 * cap the systems are factored in more, smaller batches.  KVB_MAP_PAIR=0, KVB_MAP_PAIR_STATIC=1,
 * KVB_MAP_FUSED_STRIP=0, KVB_STATS_PAIR=0, KVB_SOLVE_PERSIST=0 and
 * KVB_STATS_TC_F32=0 select the slower comparison kernels (single-CTA map,
 * fixed tile-per-pair map, separate strip pass, single-CTA statistics,
 * per-tile solver updates, CUDA-core statistics for fp32 caches); results
 * agree with the defaults within rounding.
 *
 * Checked build: the same library compiled with KVB_CHECK_BOUNDS=1
 * (libkvb_checked.so) checks the index range of every CUDA-core global access
 * of the hot kernels before it happens; a failed check skips the access and
 * the next call on the context returns KVB_ERR_CUDA.
 */
#ifndef KVB_H
#define KVB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVB_OK = 0,
    KVB_ERR_INVALID_ARG = 1,    /* null pointer, bad size, bad selection, misaligned pointer */
    KVB_ERR_SHAPE_MISMATCH = 2, /* source and target KV heads / head dims differ */
    KVB_ERR_UNSUPPORTED = 3,    /* interleaved RoPE, rope_scaling, odd head_dim, dtype */
    KVB_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed */
    KVB_ERR_NUMERIC = 5,        /* a system was not positive definite, or non-finite data */
    KVB_ERR_OOM = 6,            /* device allocation failed */
    KVB_ERR_TIMEOUT = 7         /* a bounded device wait gave up */
} kvb_status;

typedef enum { KVB_F32 = 0, KVB_BF16 = 1 } kvb_dtype;

/* One model's KV geometry ("KVBridge" ModelSignature; VeloxQuant ModelKVSpec). */
typedef struct {
    int32_t n_layers;
    int32_t n_kv_heads;
    int32_t head_dim;
    double rope_theta;
    int32_t rope_interleaved; /* 1 = interleaved ("traditional") pairs: refused */
    int32_t rope_scaling;     /* 1 = any rope_scaling: refused */
} kvb_model_spec;

typedef struct kvb_ctx kvb_ctx;
typedef struct kvb_stats kvb_stats;

/* Message of the last failed call on this thread ("" if none).  Never NULL. */
const char* kvb_last_error(void);

/* Library version, (major << 16) | minor. */
int32_t kvb_version(void);

/*
 * Create a context for one (source, target) pair on CUDA device `device`.
 * Refusals ("Cross-Model KV Transfer", "The honesty crux" item 7): mismatched
 * KV heads or head_dim -> KVB_ERR_SHAPE_MISMATCH; interleaved RoPE or
 * rope_scaling -> KVB_ERR_UNSUPPORTED; odd head_dim -> KVB_ERR_UNSUPPORTED.
 * top_k in [1, src->n_layers]; max_pos >= 1 sizes the RoPE tables.
 * Builds both cos/sin tables (float64 angle reduction) and waits for them.
 */
kvb_status kvb_ctx_create(const kvb_model_spec* src, const kvb_model_spec* tgt, int32_t top_k,
                          int32_t max_pos, int32_t device, kvb_ctx** out);

/* Free everything the context owns (syncs the device first).  NULL is a no-op. */
kvb_status kvb_ctx_destroy(kvb_ctx* ctx);

/* Pre-size the strip scratch for up to T tokens so kvb_map_apply never allocates. */
kvb_status kvb_ctx_reserve(kvb_ctx* ctx, int64_t T);

/* Sync `stream` and report (then clear) errors the kernels recorded on ctx. */
kvb_status kvb_ctx_check(kvb_ctx* ctx, void* stream);

/*
 * Kernel timing for measurement.  While enabled, every kernel the context
 * launches is bracketed by CUDA events recorded on its launch stream.
 * kvb_profile_read waits for the recorded events, writes one entry per kernel
 * name (launch count and summed device time since the last read) and clears
 * the record.  `count` receives the number of entries written (<= cap).
 */
typedef struct {
    char name[32];
    int64_t launches;
    double total_ms;
} kvb_kernel_time;

kvb_status kvb_profile_enable(kvb_ctx* ctx, int32_t on);
kvb_status kvb_profile_read(kvb_ctx* ctx, kvb_kernel_time* out, int32_t cap, int32_t* count);

/*
 * Map a source cache into a target cache ("Cross-Model KV Transfer", "The
 * mapping"; "KV-Cache zwischen Qwen3-Modellen ...", map_cache sketch).
 *   dtype       KVB_BF16: bf16 caches and W, fp32 accumulation, bf16 output
 *                         (round to nearest even); KVB_F32: fp32 caches, W and
 *                         output.  With head_dim 128 and H*d a multiple of 256
 *                         both run on the tensor cores; KVB_F32 then carries
 *                         every operand as a bf16 (hi, lo) pair, accumulates
 *                         hi*hi + hi*lo + lo*hi in fp32 (relative error near
 *                         2^-16 per product) and splits W on every call into
 *                         context scratch (4*(L_src*H*T*d + L_tgt*q*p) * 2
 *                         bytes in all); other shapes run fp32 on CUDA cores.
 *   src_k/src_v device [L_src][H][T][d] (keys as stored, i.e. with source RoPE)
 *   positions   device [T] int32
 *   sel_k/sel_v host   [L_tgt][k] int32, entries distinct within a row, in range
 *   W_k/W_v     device [L_tgt][H*d][k*H*d]  (dtype)
 *   b_k/b_v     device [L_tgt][H*d] float32
 *   out_k/out_v device [L_tgt][H][T][d] (dtype), fully overwritten
 * T == 0 is a no-op.  Device pointers must be 16-byte aligned.  Calls on one
 * context share its scratch (the stripped keys, the strip's work counters):
 * issue them on one stream, or order them, never overlapping on the GPU; use
 * one context per concurrent stream.
 */
kvb_status kvb_map_apply(kvb_ctx* ctx, kvb_dtype dtype, const void* src_k, const void* src_v,
                         const int32_t* positions, int64_t T, const int32_t* sel_k,
                         const int32_t* sel_v, const void* W_k, const void* W_v, const float* b_k,
                         const float* b_v, void* out_k, void* out_v, void* stream);

/*
 * kvb_map_apply_noalloc -- the pages have no counterpart; this is a deployment
 * variant of kvb_map_apply for callers that cannot allocate device memory,
 * such as code running inside another framework's caching allocator or a
 * runtime that owns the whole device budget: they cannot create a kvb_ctx,
 * because a context allocates its RoPE tables and strip scratch.
 *   Same arguments and results as kvb_map_apply (bf16 only, head_dim 128,
 *   n_kv_heads * 128 a multiple of 256), with the pair described by
 *   src / tgt / top_k / max_pos instead of a context.  The caller passes
 *   inputs and outputs; the call allocates nothing.  Its scratch (both RoPE
 *   tables, the stripped source keys, an error word) lives in a fixed 64 MiB
 *   array inside the library, held on every GPU that loads the library until
 *   the process exits.
 *   Limit: 8*max_pos*head_dim + 2*L_src*n_kv_heads*T*head_dim bytes (plus
 *   alignment) must fit in 64 MiB, else KVB_ERR_INVALID_ARG; e.g. about 800
 *   tokens at the Qwen3-14B -> 32B shape with max_pos = T.
 *   The first call on each device looks up the array's device address with
 *   cudaGetSymbolAddress (again after that device's context is re-created,
 *   e.g. by cudaDeviceReset); make that first call before capturing a stream.
 *   Every call reuses the same array, so calls that overlap on the GPU (other
 *   streams, other host threads) race: serialise them.  The call waits for its
 *   own kernels on `stream` and returns their errors (bad position, timeout).
 *   It reads KVB_WAIT_TIMEOUT_MS on every call.
 */
kvb_status kvb_map_apply_noalloc(const kvb_model_spec* src, const kvb_model_spec* tgt, int32_t top_k,
                                 int32_t max_pos, const void* src_k, const void* src_v,
                                 const int32_t* positions, int64_t T, const int32_t* sel_k,
                                 const int32_t* sel_v, const void* W_k, const void* W_v,
                                 const float* b_k, const float* b_v, void* out_k, void* out_v,
                                 void* stream);

/*
 * Calibration statistics ("KVBridge" README, "Loading").  One object holds, for
 * K and for V, the observation count n, the feature and target means, the
 * centered Gram over ALL source features (L_src*H*d square), the centered
 * cross statistics against ALL target columns (L_src*H*d x L_tgt*H*d) and the
 * per-column target sum of squares, all float32.  Per-target statistics for
 * any selection are sub-blocks of these (centering commutes with choosing
 * columns).  max_batch_tokens bounds T of one kvb_stats_accumulate call.
 */
kvb_status kvb_stats_create(kvb_ctx* ctx, kvb_dtype dtype, int64_t max_batch_tokens,
                            kvb_stats** out);

/*
 * Target-layer block ("KVBridge" README, "Loading": target-layer blocking
 * bounds peak memory at the cost of more passes over the calibration data).
 * The object holds the statistics of target layers [t_begin, t_end) only:
 * the full-source Gram as above, but the cross statistics, target means and
 * target sums of squares of the block's (t_end - t_begin)*H*d columns, so the
 * memory is 4 * (L_src*H*d)^2 + 4 * L_src*H*d * (t_end - t_begin)*H*d bytes
 * per kv instead of the full L_tgt*H*d columns.  kvb_stats_accumulate still
 * takes the whole [L_tgt][H][T][d] target caches and reads the block's layers;
 * kvb_layer_select writes (and kvb_ridge_solve reads) only the block's rows
 * of the selections, R^2, W and b; export / import move the block's columns.
 * A fit over all target layers runs one pass over the calibration data per
 * block.  kvb_stats_create is the block [0, L_tgt).  Requires
 * 0 <= t_begin < t_end <= L_tgt (else KVB_ERR_INVALID_ARG).
 */
kvb_status kvb_stats_create_block(kvb_ctx* ctx, kvb_dtype dtype, int64_t max_batch_tokens,
                                  int32_t t_begin, int32_t t_end, kvb_stats** out);
kvb_status kvb_stats_destroy(kvb_stats* st);

/* Zero the statistics (n = 0), asynchronously on `stream`. */
kvb_status kvb_stats_reset(kvb_stats* st, void* stream);

/*
 * Fold one batch of calibration tokens into `st` with a Chan merge.
 *   src_k/src_v device [L_src][H][T][d], tgt_k/tgt_v device [L_tgt][H][T][d]
 *   (dtype of the statistics object; keys as stored, with RoPE), positions
 *   device [T].  Tokens with pos % stride == 0 are kept ("Cross-Model KV
 *   Transfer", "Configuration": stride 4).  Keys are stripped with their own
 *   model's theta; values are used raw.
 */
kvb_status kvb_stats_accumulate(kvb_ctx* ctx, kvb_stats* st, const void* src_k, const void* src_v,
                                const void* tgt_k, const void* tgt_v, const int32_t* positions,
                                int64_t T, int32_t stride, void* stream);

/* Observation count so far (syncs `stream`). */
kvb_status kvb_stats_count(kvb_stats* st, int64_t* n_obs, void* stream);

/*
 * Checkpoint and inspection of the statistics of one kv (0 = K, 1 = V):
 * device float32 buffers mean_x [L_src*H*d], mean_y [L_tgt*H*d], gram
 * [L_src*H*d]^2 (full symmetric matrix), cross [L_src*H*d][L_tgt*H*d], syy
 * [L_tgt*H*d].  Export: any buffer may be NULL to skip it; n_obs (host, may
 * be NULL) receives the count and makes the call sync `stream`.  Import
 * replaces the statistics of that kv and sets the shared count to n_obs
 * (syncs); accumulating afterwards continues with Chan merges, so a fit can
 * resume from a checkpoint.
 */
kvb_status kvb_stats_export(kvb_stats* st, int32_t kv, int64_t* n_obs, float* mean_x, float* mean_y,
                            float* gram, float* cross, float* syy, void* stream);
kvb_status kvb_stats_import(kvb_stats* st, int32_t kv, int64_t n_obs, const float* mean_x,
                            const float* mean_y, const float* gram, const float* cross,
                            const float* syy, void* stream);

/*
 * Head-averaged single-source R^2 and top-k ("KVBridge" README, "What ships").
 * For each kv in {K, V}, source layer s and target layer t: the ridge fit of
 * target t from source s alone (lambda absolute, centered), per-column
 * SSE = S_yy - diag(C^T W) - lambda diag(W^T W), per-head pooled
 * R^2_h = 1 - sum SSE / sum S_yy over the head's d columns, averaged over heads.
 * Top-k per target by (R^2 descending, source index ascending), written in
 * ascending order to sel_k_host / sel_v_host [L_tgt][k].  r2 (device, float32
 * [2][L_tgt][L_src], K first) may be NULL.  Syncs `stream`.
 */
kvb_status kvb_layer_select(kvb_ctx* ctx, kvb_stats* st, double lambda, int32_t* sel_k_host,
                            int32_t* sel_v_host, float* r2, void* stream);

/*
 * Ridge solve per target layer ("KVBridge" README, "Loading"): with the
 * centered statistics gathered for the selection, W = (M + lambda I)^-1 C and
 * b = ybar - xbar W.  W_k/W_v device [L_tgt][H*d][k*H*d] in w_dtype (float32
 * solve, rounded once on output for KVB_BF16), b_k/b_v device [L_tgt][H*d]
 * float32.  Syncs `stream`; returns KVB_ERR_NUMERIC if a system is not
 * positive definite.
 */
kvb_status kvb_ridge_solve(kvb_ctx* ctx, kvb_stats* st, const int32_t* sel_k_host,
                           const int32_t* sel_v_host, double lambda, kvb_dtype w_dtype, void* W_k,
                           void* W_v, float* b_k, float* b_v, void* stream);

/*
 * Attention-output cosine, a quality diagnostic for a mapped cache ("KVBridge"
 * README, "Real-model T2 evidence": gate on its mean and minimum; "Scope and
 * limitations", and "Cross-Model KV Transfer", "The honesty crux" item 6: it
 * tracks downstream retention where the calibration R^2 does not).  For every
 * target layer l, query head hq and query i:
 *     o_x = sum over visible j of softmax_j(q_i . k_x[j] / sqrt(d)) v_x[j]
 * for cache x in {a, b}, and cos_out[l][hq][i] = o_a . o_b / (|o_a| |o_b|)
 * (0 where either output is zero).  Query head hq reads KV head
 * hq / (n_q_heads / H) (grouped-query attention); key j is visible to query
 * i iff kv_pos[j] <= q_pos[i], so one call covers one sequence.
 *   q        device [L_tgt][n_q_heads][Tq][d] in dtype (post-RoPE queries)
 *   q_pos    device int32 [Tq]
 *   k_a, v_a device [L_tgt][H][T][d] in dtype: the cache under test
 *   k_b, v_b device, same shape: the reference cache
 *   kv_pos   device int32 [T]
 *   cos_out  device float32 [L_tgt][n_q_heads][Tq], written in full
 * Geometry (L_tgt, H, d) comes from the context's target model; d must be
 * 16, 32, 64 or 128 and n_q_heads a multiple of H.  With T = 0 the cache
 * pointers may be NULL and every cosine is 0; with Tq = 0 nothing is read.
 * KVB_BF16 with d = 128 runs on the tensor cores (exact bf16 products, fp32
 * accumulation, probabilities carried as a bf16 pair: ~16 significant bits);
 * everything else in fp32 on CUDA cores.  Asynchronous on `stream`.
 */
kvb_status kvb_attention_cosine(kvb_ctx* ctx, kvb_dtype dtype, const void* q, int32_t n_q_heads,
                                const int32_t* q_pos, int64_t Tq, const void* k_a, const void* v_a,
                                const void* k_b, const void* v_b, const int32_t* kv_pos, int64_t T,
                                float* cos_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVB_H */
