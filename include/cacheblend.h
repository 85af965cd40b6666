/*
 * cacheblend.h — C ABI of the GB300 (sm_103a) CacheBlend per-layer KV blend.
 *
 * CacheBlend reuses KV caches that were computed for each retrieved chunk on
 * its own. Per transformer layer the blend (1) moves every cached key from its
 * chunk-local RoPE position to its position in the concatenated request,
 * (2) scores each candidate token by the squared L2 distance between its
 * recomputed and its cached V, (3) keeps the k highest-scoring tokens (the
 * high-KV-deviation, HKVD, tokens) under the gradual filter, (4) splices their
 * recomputed K/V into the reused cache and (5) runs causal grouped-query
 * attention for the HKVD tokens and the query suffix over the fused cache.
 *
 * Sources (web pages):
 *   "数学推导" (CacheBlend appendix C, math derivations):
 *      §RoPE 位置编码的相对位置不变性证明  RoPE rotation R_p, R_m^T R_n = R_{n-m}
 *      §CacheBlend 中的应用              k_new = R_{p_new - p_old} k_old
 *      §问题定义 / §形式化                old/new KV in R^{n x d}, budget k, fused KV
 *      §近似解                           S = TopK_i ||V_new[i] - V_old[i]||_2^2
 *   "rag的kvcache问题":
 *      §渐进式过滤机制                    r1% at layer 1, r2% at layer 2, stable set after
 *      §独立编码                         chunk caches computed independently
 *      §transformer训练与推理并行计算的差异  causal mask
 *      §阶段二                           attention rows are independent
 *
 * Conventions for every call:
 *   - Tensors are bf16, row-major [token, head, dim] ("NHD"), contiguous, on
 *     the current CUDA device; every bf16 tensor pointer must be 16-byte
 *     aligned. Index arrays are int32 on the device.
 *   - The caller owns every tensor. The library owns only what a cb_plan holds
 *     (RoPE cos/sin table, device error word, per-layer scratch); no call
 *     other than cb_plan_create / cb_plan_destroy allocates or frees memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Every compute
 *     call only enqueues work on it and returns without synchronising.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns CB_ERR_INVALID_ARG (or CB_ERR_UNSUPPORTED) and
 *     launches nothing. Problems only the device can see (an index out of
 *     range, an unsorted list, a wait that ran out of time) skip the offending
 *     work, never fault, and are recorded in the plan's device error word,
 *     which cb_check() reads.
 *   - Sizes of 0 are valid and launch nothing.
 *   - cb_last_error_string() describes the last failure of this thread.
 */
#ifndef CACHEBLEND_H
#define CACHEBLEND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cb_status {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape: nothing launched */
  CB_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels implement (e.g. head_dim) */
  CB_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  CB_ERR_TIMEOUT = 4,      /* a device-side wait gave up (reported by cb_check) */
  CB_ERR_DEVICE_CHECK = 5  /* a device-side argument check failed (reported by cb_check) */
} cb_status;

/* Which coordinates of a head form RoPE pair j (the pages do not fix it). */
typedef enum cb_rope_style {
  CB_ROPE_HALF = 0,        /* (j, j + D/2): GPT-NeoX / Llama / Mistral layout */
  CB_ROPE_INTERLEAVED = 1  /* (2j, 2j + 1) */
} cb_rope_style;

/* What the HKVD selection ranks. */
typedef enum cb_deviation {
  CB_DEV_V = 0,  /* ||V_new - V_old||^2 ("数学推导" §近似解) */
  CB_DEV_KV = 1  /* ||K~_new - K~_old||^2 + ||V_new - V_old||^2: the deviation on the whole KV of
                    "rag的kvcache问题" §核心发现, keys compared at the same position (below) */
} cb_deviation;

/* Which tokens a layer after layer 2 chooses from ("rag的kvcache问题" §渐进式过滤机制
 * fixes layers 1 and 2; later layers are read two ways). */
typedef enum cb_filter {
  CB_FILTER_KEEP = 0,     /* layer >= 3 keeps S_{l-1} whole: no deviation, no top-k */
  CB_FILTER_RESELECT = 1  /* every layer >= 2 ranks the layer-1 pool S_1 by its own deviation, keeps k_2 */
} cb_filter;

/* One blend request: n_chunks cached chunks of chunk_len tokens (chunk-local
 * positions 0 .. chunk_len-1), then n_suffix uncached query tokens. Token i of
 * the request sits at global position i. r1_pct / r2_pct: gradual-filter
 * ratios in percent of the n_ctx = n_chunks * chunk_len cached tokens. */
typedef struct cb_config {
  int32_t n_chunks;
  int32_t chunk_len;
  int32_t n_suffix;
  int32_t hq;          /* query heads */
  int32_t hkv;         /* kv heads; hq % hkv == 0 and hq / hkv in {1,2,4,8,16} */
  int32_t head_dim;    /* 64 or 128 */
  double rope_theta;   /* RoPE base: pair j turns by p * theta^(-2j/D) */
  int32_t rope_style;  /* cb_rope_style */
  int32_t r1_pct;      /* layer-1 keep ratio, 0..100 */
  int32_t r2_pct;      /* keep ratio from layer 2 on, 0..r1_pct */
  int32_t deviation;   /* cb_deviation */
  int32_t filter;      /* cb_filter */
} cb_config;

typedef struct cb_plan cb_plan;

/* Create a plan on the current device: copies *cfg, builds the RoPE cos/sin
 * table for positions 0 .. n_tokens-1 on the host (angle p * theta^(-2j/D) in
 * fp64 with the C library's pow, cos and sin, rounded to fp32) and copies it
 * to the device, and creates the device error word and the side streams of
 * cb_blend_request. Synchronous. */
cb_status cb_plan_create(const cb_config* cfg, cb_plan** out);

/* Free everything the plan owns. Waits for the device first. NULL is a no-op. */
cb_status cb_plan_destroy(cb_plan* plan);

/* Sizes of layer `layer` (1-based) under the plan's gradual filter:
 * n_cand = |C_l| (candidates read), k = |S_l| (kept), mq = k + n_suffix
 * (attention query rows), selects = 1 if the layer runs deviation + top-k.
 * Layer 1: C = all n_ctx tokens, k = floor(r1 * n_ctx / 100). Layer 2: C = S_1,
 * k = floor(r2 * n_ctx / 100). Layer >= 3: C = S_{l-1}, kept whole
 * (CB_FILTER_KEEP), or C = S_1 and k = floor(r2 * n_ctx / 100) selected again
 * (CB_FILTER_RESELECT). */
cb_status cb_layer_sizes(const cb_plan* plan, int32_t layer, int32_t* n_cand, int32_t* k,
                         int32_t* mq, int32_t* selects);

/* RoPE row rotation ("数学推导" §RoPE 位置编码的相对位置不变性证明 and
 * §CacheBlend 中的应用):
 *   out[out_rows ? out_rows[i] : i] = R_{pos_to[i] - (pos_from ? pos_from[i] : 0)} x[in_rows ? in_rows[i] : i]
 * for i in [0, n). Each row is n_heads x head_dim (the plan's) bf16; math in
 * fp32 with the plan's cos/sin table. pos_from == NULL encodes at pos_to
 * (k~ = R_p k); otherwise it re-rotates a key cached at pos_from to pos_to.
 * |pos_to - pos_from| must be < n_tokens of the plan (else the row is skipped
 * and CB_ERR_DEVICE_CHECK is recorded). x holds x_rows rows and out holds
 * out_rows_total rows; a mapped row outside them is skipped and recorded the
 * same way. pos_to must not be NULL. out may equal x only when in_rows and
 * out_rows are both NULL (in place). */
cb_status cb_rope_rerotate(cb_plan* plan, void* out, const void* x, const int32_t* in_rows,
                           const int32_t* out_rows, const int32_t* pos_from, const int32_t* pos_to,
                           int32_t n, int32_t n_heads, int32_t x_rows, int32_t out_rows_total,
                           void* stream);

/* V deviation ("数学推导" §近似解): for i in [0, m),
 *   dev[i] = sum_{h, j} (v_new[t, h, j] - v_old[t, h, j])^2,  t = cand ? cand[i] : i,
 * in fp32 in one fixed order (8-element chunks dealt to 32 lanes, sequential
 * per lane, then a xor butterfly over lanes 16, 8, 4, 2, 1; products and sums
 * rounded separately, no fused multiply-add), so the value is reproducible
 * bit for bit. v_new and v_old are indexed by token ([>= t+1, hkv, D]).
 * Candidates outside [0, n_ctx) are skipped (dev = NaN, CB_ERR_DEVICE_CHECK). */
cb_status cb_kv_deviation(cb_plan* plan, const void* v_new, const void* v_old, const int32_t* cand,
                          int32_t m, float* dev, void* stream);

/* K+V deviation (CB_DEV_KV): for i in [0, m), t = cand ? cand[i] : i,
 *   dev[i] = sum_{h,j} (R_{p_new} k_new[t] - R_{p_new - p_old} k_old[t])[h,j]^2
 *          + sum_{h,j} (v_new[t, h, j] - v_old[t, h, j])^2,
 * with p_old = t mod chunk_len (the cached key's chunk-local position) and
 * k_new the recomputed key before RoPE. Rotations keep lengths, so the key
 * term is computed as ||R_{p_old} k_new[t] - k_old[t]||^2 (one turn): each
 * element of R_{p_old} k_new in fp32 from the plan's table row p_old, first
 * pair member fl(fl(x c) - fl(y s)), second fl(fl(x s) + fl(y c)), then the
 * canonical order of cb_kv_deviation over the sequence [key part padded to a
 * multiple of 256 elements, V part padded the same way]: every lane adds its
 * key chunks, then its V chunks. Same layouts and error behaviour as
 * cb_kv_deviation; k_new / k_old [>= t+1, hkv, D] by token. */
cb_status cb_kv_deviation_kv(cb_plan* plan, const void* k_new, const void* k_old, const void* v_new,
                             const void* v_old, const int32_t* cand, int32_t m, float* dev, void* stream);

/* HKVD top-k ("数学推导" §近似解; gradual filter of "rag的kvcache问题"
 * §渐进式过滤机制): keep the k of m candidates with the largest dev, ties to
 * the lower token id. cand (NULL = identity) must be strictly ascending.
 * Writes sel_tok[k] (ascending token ids) and sel_row[k] (their indices in
 * cand). dev values must not be NaN. One thread block; no scratch memory. */
cb_status cb_hkvd_topk(cb_plan* plan, const float* dev, const int32_t* cand, int32_t m, int32_t k,
                       int32_t* sel_tok, int32_t* sel_row, void* stream);

/* Fuse / scatter ("数学推导" §形式化): for each token t of sel_tok[0..k) and
 * each suffix token t in [n_ctx, n_tokens):
 *   k_fused[t] = R_t k_new[t],  v_fused[t] = v_new[t]
 * leaving every other row of k_fused / v_fused untouched. k_new / v_new are
 * token-indexed [n_tokens, hkv, D]; k_fused / v_fused are [n_tokens, hkv, D].
 * sel_tok must be strictly ascending context token ids. */
cb_status cb_fuse_scatter(cb_plan* plan, void* k_fused, void* v_fused, const void* k_new,
                          const void* v_new, const int32_t* sel_tok, int32_t k, void* stream);

/* HKVD causal GQA attention ("数学推导" §形式化; causal mask of
 * "rag的kvcache问题" §transformer训练与推理并行计算的差异):
 *   out[i, h] = sum_{j <= q_pos[i]} softmax_j(scale * q[i, h] . k[j, g]) v[j, g],  g = h / (hq/hkv)
 * q, out: [mq, hq, D] compact query rows already RoPE-encoded at q_pos;
 * k, v: [n_keys, hkv, D], key j at position j. q_pos strictly ascending,
 * each < n_keys (a violation is recorded, rows still bounded). scale <= 0
 * selects 1/sqrt(D). fp32 accumulation and softmax, bf16 P, bf16 output.
 * tcgen05 (TMEM accumulators) fed by TMA. */
cb_status cb_hkvd_attention(cb_plan* plan, const void* q, const int32_t* q_pos, int32_t mq,
                            const void* k, const void* v, int32_t n_keys, float scale, void* out,
                            void* stream);

/* QKV projection of the rows a layer recomputes ("rag的kvcache问题" §阶段一: each token's q, k,
 * v is its hidden vector times the projection weights, computed as one product of the stacked
 * rows; §渐进式过滤机制: at a layer only the candidate tokens and the suffix are recomputed):
 *   y_i = x[t] W^T,  t = rows ? rows[i] : i,  i in [0, m),
 *   q[t] = y_i[Q heads], k[t] = y_i[K heads], v[t] = y_i[V heads]  (bf16),
 * with q and k RoPE-encoded at position t (the plan's table and style) when `encode` != 0, and
 * left before RoPE otherwise (the form cb_blend_layer reads as k_new / q). x: [x_rows, d_model]
 * bf16 hidden rows, d_model a positive multiple of 64 (else CB_ERR_UNSUPPORTED). w_qkv:
 * [(hq + 2 hkv) D, d_model] bf16, one output feature per row (Q heads, then K heads, then V
 * heads). q: [n_tokens, hq, D], k, v: [n_tokens, hkv, D] of the plan, written only at the rows'
 * tokens. With a row list, x_gathered (caller-owned, [m, d_model] bf16) receives the gathered rows
 * first; NULL rows read x[0 .. m) in place. A row outside x (or past n_tokens) is recorded as
 * CB_ERR_DEVICE_CHECK and not written. tcgen05 GEMM (bf16 in, fp32 accumulate) fed by TMA. */
cb_status cb_qkv_projection(cb_plan* plan, const void* x, int32_t x_rows, int32_t d_model, const int32_t* rows,
                            int32_t m, const void* w_qkv, int32_t encode, void* x_gathered, void* q, void* k, void* v,
                            void* stream);

/* The same projection with the row of x and the token written given separately (the layout of a
 * layer-by-layer pass, "rag的kvcache问题" §渐进式过滤机制: the hidden rows a layer passes on are those
 * of the tokens it recomputed, in its list order, so the next layer reads them in place when its
 * set is the same, and by position in that list when its set is a subset):
 *   y_i = x[x_index ? x_index[i] : i] W^T,  written (and RoPE-encoded) at token
 *   t_i = tokens ? tokens[i] : i,  i in [0, m).
 * cb_qkv_projection(rows) is x_index = tokens = rows. With x_index, x_gathered (caller-owned,
 * [m, d_model] bf16) receives the gathered rows first; without it x[0 .. m) is read in place
 * (m <= x_rows). Without tokens, m <= n_tokens. An index outside x, or a token outside the plan's
 * n_tokens, is recorded as CB_ERR_DEVICE_CHECK and that row is not written. */
cb_status cb_qkv_projection_indexed(cb_plan* plan, const void* x, int32_t x_rows, int32_t d_model,
                                    const int32_t* x_index, const int32_t* tokens, int32_t m, const void* w_qkv,
                                    int32_t encode, void* x_gathered, void* q, void* k, void* v, void* stream);

/* Decode attention over a cache ("rag的kvcache问题" §阶段 2 (Decode): after the prefill the
 * newest token is the only query, and its [1, d] query row is matched against the whole
 * cached K/V, which makes the step memory-bound). For the newest token at position
 * n_keys - 1, with its own key and value already in the cache's last row:
 *   out[h] = sum_{j < n_keys} softmax_j(scale * q[h] . k[j, g]) v[j, g],  g = h / (hq/hkv),
 * q, out: [hq, D] (q RoPE-encoded at n_keys - 1); k, v: [n_keys, hkv, D], key j at
 * position j (e.g. a layer's k_fused / v_fused with the new token appended). scale <= 0
 * selects 1/sqrt(D). Both products run on the tensor cores (bf16 in, fp32 accumulate; the
 * softmax weights rounded to bf16 before P V, as in cb_hkvd_attention); bf16 output. The keys
 * of each kv head are split over up to 40 CTAs (one wave over all kv heads) whose partial
 * results meet in the plan's decode scratch (the last CTA of a kv head merges them), so decode
 * calls on one plan must not overlap on the GPU: order them on one stream, or give each stream
 * its own plan. A bounded wait that gives up records CB_ERR_TIMEOUT in the plan's error word. */
cb_status cb_decode_attention(cb_plan* plan, const void* q, const void* k, const void* v, int32_t n_keys,
                              float scale, void* out, void* stream);

/* Attention sparsity ("数学推导" §注意力稀疏性的量化分析: Sparsity(A, eps) =
 * |{(i, j): A_ij < eps}| / n^2 for the attention weights A): for the causal attention of
 * cb_hkvd_attention (same q, q_pos, k, v, n_keys, scale; masked keys have weight 0 and count),
 * counts the weights below eps of every query row and head over all n_keys keys:
 *   counts[i * hq + h] = |{j < n_keys: A[h]_ij < eps}|,  *total = sum of counts (uint64).
 * Two launches of the attention kernel: the first writes out (as cb_hkvd_attention) and
 * row_stats ([mq, hq] float2: a reference r in log2 units and the sum s of 2^(score - r), so
 * that the row's softmax denominator is s * 2^r; r lies at most 16 below the row's largest
 * scaled score), the second recomputes the same scores and compares them with r + log2(eps * s);
 * then a reduction writes *total.
 * Sparsity = total / (hq * mq * n_keys) (with q_pos = 0 .. n - 1 and n_keys = n this is the
 * page's n x n figure summed over heads). eps must be positive. Weights within about 1e-5 of eps
 * (relative) may fall on either side of it (fp32 scores and softmax sums). */
cb_status cb_attention_sparsity(cb_plan* plan, const void* q, const int32_t* q_pos, int32_t mq, const void* k,
                                const void* v, int32_t n_keys, float scale, float eps, void* out, void* row_stats,
                                int32_t* counts, uint64_t* total, void* stream);

/* Attention deviation ("数学推导" §形式化: ||Attention(Q, K_fused, V_fused) -
 * Attention(Q, K_new, V_new)||, the objective the HKVD selection approximates): over `rows`
 * rows of [hq, D] bf16 outputs, sums[0] = sum (o - o_ref)^2 and sums[1] = sum o_ref^2 in fp64
 * (device memory, overwritten). The Frobenius norms are their square roots. The blocks' partial
 * sums are added in no fixed order, so the last bits can differ between runs. */
cb_status cb_output_deviation(cb_plan* plan, const void* o, const void* o_ref, int32_t rows, double* sums,
                              void* stream);

/* Buffers of one layer for cb_blend_layer. Sizes from cb_layer_sizes. */
typedef struct cb_layer_io {
  const void* k_old;     /* [n_ctx, hkv, D] cached keys, at chunk-local positions */
  const void* v_old;     /* [n_ctx, hkv, D] cached values */
  const void* k_new;     /* [n_tokens, hkv, D] recomputed keys before RoPE, by token; rows of C_l and the suffix are read */
  const void* v_new;     /* [n_tokens, hkv, D] recomputed values, by token; same rows */
  const void* q;         /* [n_tokens, hq, D] queries before RoPE, by token; rows of S_l and the suffix are read */
  const int32_t* cand;   /* C_l, strictly ascending: NULL at layer 1 (all context tokens), else S_{l-1}
                            (CB_FILTER_RESELECT: S_1) */
  float* dev;            /* [n_cand] out at selecting layers: deviation per candidate (may be NULL otherwise) */
  int32_t* sel_tok;      /* [k] out: S_l, ascending token ids */
  int32_t* sel_row;      /* [k] out: rows of S_l in C_l */
  void* k_fused;         /* [n_tokens, hkv, D] out: fused keys at global positions */
  void* v_fused;         /* [n_tokens, hkv, D] out: fused values */
  void* q_rot;           /* [mq, hq, D] out: encoded query rows (S_l, then the suffix) */
  void* out;             /* [mq, hq, D] out: attention output rows, same order */
} cb_layer_io;

/* One layer of the blend (1-based `layer`), all on `stream`, no host sync:
 *   selecting layers: deviation over C_l (V or K+V, as the plan's config
 *                     says), then top-k -> S_l;
 *   other layers:     S_l = C_l;
 *   then fused K/V for all n_tokens rows in one pass (cached rows re-rotated
 *   by their chunk offset, S_l and suffix rows encoded from k_new / v_new)
 *   with the query rows encoded in the same launch, and the attention. */
cb_status cb_blend_layer(cb_plan* plan, int32_t layer, const cb_layer_io* io, void* stream);

/* All layers 1..n_layers of one request (ios[l-1] = buffers of layer l) with
 * the gradual filter wired automatically: layer l reads the candidates
 * ios[l-2].sel_tok (CB_FILTER_RESELECT: ios[0].sel_tok for l >= 2; ios[].cand
 * is ignored). Same results as calling
 * cb_blend_layer for each layer in order, but scheduled over streams the plan
 * owns: every layer's deviation, top-k and fused-cache (with query encoding)
 * kernels run on one side stream, ahead of the attention, and the attention of
 * consecutive layers runs on two streams, so that one layer's attention
 * overlaps the next layer's streaming kernels and the tail of the previous
 * attention. All work is ordered after prior work on `stream` and completes
 * before later work on it. The layers' buffers must not alias one another.
 * Capturable into a CUDA graph on `stream`. */
cb_status cb_blend_request(cb_plan* plan, int32_t n_layers, const cb_layer_io* ios, void* stream);

/* The stages of one layer, in the order cb_blend_layer runs them. */
typedef enum cb_stage {
  CB_STAGE_DEVIATION = 0, /* deviation over C_l (selecting layers only) */
  CB_STAGE_TOPK = 1,      /* top-k of the deviations -> S_l (selecting layers only) */
  CB_STAGE_FUSE = 2,      /* fused K/V for all n_tokens rows and the encoded query rows, one launch */
  CB_STAGE_ATTENTION = 3  /* HKVD attention */
} cb_stage;

/* One stage of cb_blend_layer alone, on `stream`: the kernel cb_blend_layer
 * launches for that stage, reading what the earlier stages of the same layer
 * wrote into `io` (run the stages in order, or after a cb_blend_layer of the
 * layer). A stage the layer does not have (deviation and top-k at layers that
 * keep their candidates) is a no-op returning CB_OK. Every stage is
 * idempotent: it rewrites the same outputs from the same inputs. For timing
 * or profiling one kernel type at a time; capturable into a CUDA graph. */
cb_status cb_blend_stage(cb_plan* plan, int32_t layer, const cb_layer_io* io, int32_t stage, void* stream);

/* HKVD selection that allocates nothing (the pages have no counterpart: this
 * is a deployment aid). For callers that cannot allocate device memory where
 * they select tokens, e.g. a serving engine whose own pool owns all free HBM
 * (a cudaMalloc there fails or fragments the pool), or a latency-critical
 * path that cannot pay cudaMalloc's implicit device synchronisation; such a
 * caller cannot create a cb_plan either. Computes exactly what
 * cb_kv_deviation followed by cb_hkvd_topk compute (same kernels, same
 * fixed-order fp32 deviation, same tie rule), without a plan:
 *   v_new, v_old  [>= n_rows, hkv, head_dim] bf16, token-indexed, 16-B aligned
 *   cand          [m] strictly ascending token ids < n_rows, or NULL (= 0..m-1)
 *   sel_tok/row   [k] outputs, as cb_hkvd_topk.
 * The per-candidate deviations live in one array compiled into the library,
 * CB_NOALLOC_MAX_CANDIDATES floats (256 KiB) on every GPU that loads it,
 * held until the process exits; m above that limit returns
 * CB_ERR_INVALID_ARG. The first call on a device looks up that array's device
 * address (with the device current) and remembers it with the ID of the
 * CUDA context it belongs to; a call that finds another context current on
 * the device (after cudaDeviceReset, say) looks it up again. Make the first
 * call on each device, and the first after such a reset, before any stream
 * capture. All calls share the array: calls
 * whose work overlaps on the GPU (different streams, no ordering between
 * them) race and can return wrong selections; order them on one stream.
 * Device-side argument findings are not recorded (there is no plan to hold an
 * error word): an out-of-range candidate gets a NaN deviation, which ranks
 * first. Calls no cudaMalloc, cudaFree or allocating library routine. */
#define CB_NOALLOC_MAX_CANDIDATES 65536
cb_status cb_hkvd_select_noalloc(const void* v_new, const void* v_old, const int32_t* cand, int32_t m,
                                 int32_t k, int32_t n_rows, int32_t hkv, int32_t head_dim,
                                 int32_t* sel_tok, int32_t* sel_row, void* stream);

/* Which of the two attention kernels a cb_hkvd_attention call (or a blend
 * layer's attention) of mq query rows runs on the plan's device: 1 for the
 * paired-tile kernel (two 128-row query tiles per CTA whose softmax and
 * tensor-core work alternate; head_dim 128, and only when the launch fills
 * at least 1.5 waves of the GPU's SMs), 0 for the one-tile kernel. Both
 * compute the same attention; the answer is for profiling and tests. */
int32_t cb_attention_uses_paired_tiles(const cb_plan* plan, int32_t mq);

/* Test support for the failure path, not part of the blend (the pages have
 * no counterpart). Runs cb_hkvd_attention's kernel (head_dim 128 only) in a
 * form whose K-tile producer never requests key tile 1 and whose bounded
 * waits give up after 100 us instead of 2 s: every CTA whose queries reach
 * that tile (a query position >= 128) records CB_ERR_TIMEOUT in the plan's
 * error word, skips its remaining rounds, waits (again bounded) for its own
 * copies and tensor-core work, frees its tensor memory and returns, leaving
 * its rows of `out` unwritten. The next cb_check reports CB_ERR_TIMEOUT and
 * clears the word, and the device stays usable. Arguments as
 * cb_hkvd_attention; CB_ERR_INVALID_ARG if n_keys <= 128 or mq <= 0. */
cb_status cb_test_attention_wait_timeout(cb_plan* plan, const void* q, const int32_t* q_pos, int32_t mq,
                                         const void* k, const void* v, int32_t n_keys, void* out, void* stream);

/* Test support for the failure path, not part of the blend (the pages have no
 * counterpart). Runs cb_decode_attention's kernel (head_dim 128 only) in a form
 * whose producer never copies key tile 1 of its split and whose bounded waits
 * give up after 100 us instead of 2 s: every CTA with a second key tile records
 * CB_ERR_TIMEOUT in the plan's error word, skips the rest of its tiles, waits
 * (again bounded) for its own copies and tensor-core work, frees its tensor
 * memory and still takes its ticket, so the split counters stay consistent; the
 * contents of `out` are undefined. The next cb_check reports CB_ERR_TIMEOUT and
 * clears the word, and the device and the plan stay usable. Arguments as
 * cb_decode_attention (scale 1/sqrt(D)); CB_ERR_INVALID_ARG if n_keys <= 128. */
cb_status cb_test_decode_wait_timeout(cb_plan* plan, const void* q, const void* k, const void* v, int32_t n_keys,
                                      void* out, void* stream);

/* Test support for the failure path, not part of the blend (the pages have no
 * counterpart). Runs cb_qkv_projection's kernel (head_dim 128; x[0 .. m) read in
 * place, written at tokens 0 .. m-1, no RoPE) in a form where the first CTA of
 * every CTA pair arms the barrier of K step 1 for the pair's bytes but never
 * copies its own share, and every bounded wait gives up after 100 us instead of
 * 2 s: both CTAs record CB_ERR_TIMEOUT in the plan's error word, drain the MMAs
 * and copies they started, free their tensor memory and meet at the final
 * cluster barrier; q, k, v are left unwritten or partly written. The next
 * cb_check reports CB_ERR_TIMEOUT and clears the word, and the device stays
 * usable. CB_ERR_INVALID_ARG unless 0 < m <= n_tokens and d_model >= 128. */
cb_status cb_test_projection_wait_timeout(cb_plan* plan, const void* x, int32_t d_model, int32_t m,
                                          const void* w_qkv, void* q, void* k, void* v, void* stream);

/* Synchronise the plan's device, read and clear its error word. Returns
 * CB_OK, CB_ERR_TIMEOUT or CB_ERR_DEVICE_CHECK (detail in
 * cb_last_error_string). Off the hot path. */
cb_status cb_check(cb_plan* plan);

/* Human-readable description of the last failure on this thread. */
const char* cb_last_error_string(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t cb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CACHEBLEND_H */
