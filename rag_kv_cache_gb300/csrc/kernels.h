// Host-side launchers of the blend's kernels (internal to the library; the
// public interface is include/cacheblend.h). Every launcher only enqueues on
// `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cb {

// Row index map: row i -> (i < k ? (idx ? idx[i] : i) : base + (i - k)); rows at or
// beyond `limit` (the tensor's row count) are rejected by the kernel.
struct RowMap {
  const int32_t* idx;
  int32_t k;
  int32_t base;
  int32_t limit;
};

struct RopeTable {
  const float2* tab;  // [len][head_dim / 2] (cos, sin) of p * theta^(-2j/D)
  int32_t len;
};

// out[omap(i)] = R_{pos_to(i) - pos_from(i)} x[imap(i)], i in [0, n).
// pos_to == nullptr: pos_to(i) = imap(i) (encode at the token's own position).
// pos_from == nullptr: pos_from(i) = 0. pos_out (optional) receives pos_to(i).
cudaError_t launch_rope_rows(void* out, const void* x, RowMap imap, RowMap omap, const int32_t* pos_from,
                             const int32_t* pos_to, int32_t* pos_out, int32_t n, int32_t n_heads,
                             int32_t head_dim, int32_t style, RopeTable t, int32_t* err, cudaStream_t s);

// Deviation per candidate in the canonical fp32 order: V only when k_new is null, else K+V
// (the key part turned to p_old = token mod chunk_len with the table and RoPE style).
// Several layers' selections over one candidate list (the re-selection reading of the gradual
// filter: every layer >= 2 selects from S_1): one launch of deviations (a grid row per layer) and
// one of top-k (a block per layer), up to kSelectBatchMax layers. k_new / k_old null: V deviation.
constexpr int kSelectBatchMax = 16;
struct SelectBatch {
  int n;
  const void* k_new[kSelectBatchMax];
  const void* k_old[kSelectBatchMax];
  const void* v_new[kSelectBatchMax];
  const void* v_old[kSelectBatchMax];
  float* dev[kSelectBatchMax];
  int32_t* sel_tok[kSelectBatchMax];
  int32_t* sel_row[kSelectBatchMax];
};
cudaError_t launch_select_batch(const SelectBatch& b, const int32_t* cand, int32_t m, int32_t k, int32_t n_rows,
                                int32_t hkv, int32_t head_dim, int32_t chunk_len, int32_t style, RopeTable t,
                                int32_t* err, cudaStream_t s);

cudaError_t launch_kv_deviation(const void* k_new, const void* k_old, const void* v_new, const void* v_old,
                                const int32_t* cand, int32_t m, int32_t n_rows, int32_t hkv, int32_t head_dim,
                                int32_t chunk_len, int32_t style, RopeTable t, float* dev, int32_t* err,
                                cudaStream_t s);

cudaError_t launch_hkvd_topk(const float* dev, const int32_t* cand, int32_t m, int32_t k, int32_t* sel_tok,
                             int32_t* sel_row, int32_t* err, cudaStream_t s);

// Scatter encoded recomputed rows (sel_tok[0..k) and the suffix) into the fused cache.
cudaError_t launch_fuse_scatter(void* k_fused, void* v_fused, const void* k_new, const void* v_new,
                                const int32_t* sel_tok, int32_t k, int32_t n_ctx, int32_t n_tokens,
                                int32_t hkv, int32_t head_dim, int32_t style, RopeTable t, int32_t* err,
                                cudaStream_t s);

// One pass over all n_tokens rows: cached rows re-rotated by their chunk offset,
// selected and suffix rows encoded from k_new / v_new. With copy_tok set, the
// list sel_tok[0..k) is also copied to copy_tok / copy_row (= 0..k-1). With q set,
// the same launch also encodes the layer's mq query rows (row t < k is token
// sel_tok[t], row t >= k is token n_ctx + t - k; hq heads each) from the
// token-indexed q into the compact q_rot. narrow: 2-row blocks (else 8-row blocks).
cudaError_t launch_blend_fuse(void* k_fused, void* v_fused, const void* k_old, const void* v_old,
                              const void* k_new, const void* v_new, const int32_t* sel_tok, int32_t k,
                              int32_t* copy_tok, int32_t* copy_row, int32_t n_ctx, int32_t chunk_len,
                              int32_t n_tokens, int32_t hkv, int32_t head_dim, int32_t style, RopeTable t,
                              const void* q, void* q_rot, int32_t mq, int32_t hq, bool narrow, int32_t* err,
                              cudaStream_t s);


// Positions of the compact query rows: row t < k sits at idx[t], row t >= k at base + (t - k).
// wait_prior: the kernel waits for its predecessor on the stream (programmatic launch) before
// reading; false when the caller orders its inputs by events and allows the overlap.
struct QueryPositions {
  const int32_t* idx;
  int32_t k;
  int32_t base;
  bool wait_prior;
};

// Optional diagnostics of one attention launch (all null in the blend): row_stats receives each
// (row, head)'s softmax (max, sum) in log2 units; with counts set, the launch also counts per
// (row, head) the weights below 2^log2_eps over all n_keys keys, from count_stats (the row
// statistics of an earlier launch on the same inputs).
struct AttentionDiag {
  float2* row_stats = nullptr;
  const float2* count_stats = nullptr;
  float log2_eps = 0.0f;
  int32_t* counts = nullptr;
};

// Causal GQA attention over compact RoPE-encoded query rows.
cudaError_t launch_hkvd_attention(const void* q, QueryPositions qp, int32_t mq, const void* k,
                                  const void* v, int32_t n_keys, int32_t hq, int32_t hkv, int32_t head_dim,
                                  float scale, void* out, int32_t* err, cudaStream_t s,
                                  const AttentionDiag& diag = AttentionDiag());

// The two-query-tile ("ping-pong") attention kernel for large launches (attention_pp.cu):
// eligible when head_dim is 128 and the launch makes at least two waves of its 256-row CTAs;
// launch_hkvd_attention picks it then. Returns cudaErrorNotSupported, launching nothing, when
// the kernel was built with fewer registers than its warpgroups' split needs.
bool attention_pp_eligible(int32_t mq, int32_t hq, int32_t hkv, int32_t head_dim);
cudaError_t launch_hkvd_attention_pp(const void* q, QueryPositions qp, int32_t mq, const void* k, const void* v,
                                     int32_t n_keys, int32_t hq, int32_t hkv, float scale, void* out, int32_t* err,
                                     cudaStream_t s);

// The attention kernel's wait-timeout probe (test support): the same launch with head_dim 128,
// in the kernel instance whose K producer never requests key tile 1 and whose waits give up
// after 100 us. Needs n_keys > 128 (a second key tile).
cudaError_t launch_attention_timeout_probe(const void* q, QueryPositions qp, int32_t mq, const void* k,
                                           const void* v, int32_t n_keys, int32_t hq, int32_t hkv, float scale,
                                           void* out, int32_t* err, cudaStream_t s);

// Diagnostics reductions. sum_counts: *total = sum of counts[0..n) (64-bit). output_deviation:
// sums[0] = sum (a - b)^2, sums[1] = sum b^2 over n bf16 elements, in fp64 (order of the block
// partials not fixed: the last bits may differ between runs).
cudaError_t launch_sum_counts(const int32_t* counts, int64_t n, unsigned long long* total, cudaStream_t s);
cudaError_t launch_output_deviation(const void* a, const void* b, int64_t n, double* sums, cudaStream_t s);

// Scratch of the decode attention (owned by the plan): per (kv head, split, q head) an
// unnormalised output row and its (max, sum), and one ticket counter per kv head that is
// zero between calls (the kernel leaves it zero).
struct DecodeScratch {
  float* part_o;      // [hkv][decode_max_splits()][G][D]
  float2* part_ml;    // [hkv][decode_max_splits()][G]
  int32_t* tickets;   // [hkv]
  int32_t sms;        // the device's SM count (the launch takes one CTA per SM, one wave)
};

int32_t decode_max_splits();

// Decode attention on the tensor cores: one query row q [hq, D] over the whole cache k, v
// [n_keys, hkv, D] (head_dim 64 or 128, at most 32 query heads per kv head); `err` receives a
// timeout of one of its bounded waits.
bool decode_tc_supported(int32_t hq, int32_t hkv, int32_t head_dim);
cudaError_t launch_decode_tc(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq, int32_t hkv,
                             int32_t head_dim, float scale, void* out, const DecodeScratch& ws, int32_t* err,
                             cudaStream_t s);
// Test support: the same kernel (head_dim 128) in a form whose key tile 1 never arrives and whose
// waits give up after kProbeTimeoutNs (n_keys > 128).
cudaError_t launch_decode_timeout_probe(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq,
                                        int32_t hkv, float scale, void* out, const DecodeScratch& ws, int32_t* err,
                                        cudaStream_t s);

// QKV projection of listed rows: q / k / v rows of token t_i = tokens[i] (null: i) from
// x[x_index[i]] W^T (x_index null: x[i], read in place; else the rows are first copied to
// x_gathered [m, d_model]), q and k RoPE-encoded at position t_i when `encode`.
// W: [(hq + 2 hkv) head_dim, d_model].
cudaError_t launch_qkv_projection(const void* x, int32_t x_rows, int32_t d_model, const int32_t* x_index,
                                  const int32_t* tokens, int32_t m, void* x_gathered, const void* w, int32_t n_tokens,
                                  int32_t hq, int32_t hkv, int32_t head_dim, int32_t encode, int32_t style, RopeTable t,
                                  void* q, void* k, void* v, int32_t* err, cudaStream_t s);
bool qkv_projection_supported(int32_t d_model);
// Test support: the projection kernel (head_dim 128, x read in place, no RoPE) in a form whose K
// step 1 never completes and whose waits give up after kProbeTimeoutNs (d_model >= 128).
cudaError_t launch_projection_timeout_probe(const void* x, int32_t d_model, int32_t m, const void* w, int32_t n_tokens,
                                            int32_t hq, int32_t hkv, void* q, void* k, void* v, int32_t* err,
                                            cudaStream_t s);

}  // namespace cb
