// C ABI of the blend (declared in include/cacheblend.h): host-side argument
// checks, the plan (RoPE table, device error word, scratch), and the
// per-layer driver that enqueues the kernels of one layer on the caller's
// stream without any host synchronisation.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/cacheblend.h"
#include "common.cuh"
#include "kernels.h"

// Streams that run consecutive layers' attention in cb_blend_request (the caller's stream and
// CB_ATTN_STREAMS - 1 of the plan's): a layer's attention overlaps the tails of the layers before it.
#ifndef CB_ATTN_STREAMS
#define CB_ATTN_STREAMS 2
#endif
constexpr int kAttnStreams = CB_ATTN_STREAMS;
static_assert(kAttnStreams >= 1 && kAttnStreams <= 8, "attention streams");

struct cb_plan {
  cb_config cfg;
  int device;
  int32_t n_ctx;
  int32_t n_tokens;
  float2* rope_tab;  // [n_tokens][head_dim / 2]
  int32_t* err;      // [0] flags, [1] first offending index (-1 = none)
  cudaStream_t aux_stream;  // cb_blend_request: every layer's deviation, top-k and fuse (with the query encoding)
  cudaStream_t aux_attn[kAttnStreams];  // cb_blend_request: attention of layer l on stream (l - 1) % kAttnStreams
                                        // ([0] unused: that one is the caller's stream)
  cudaEvent_t ev_fork, ev_ready, ev_join;
  cb::DecodeScratch decode;  // cb_decode_attention's split partials and ticket counters
};

namespace {

// Every entry point is one NVTX range named after it, so a profile of a request reads by call
// (a push and a pop through an unset function pointer when no tool collects NVTX).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
#define CB_NVTX_RANGE() const NvtxRange cb_nvtx_range_(__func__)

thread_local std::string g_last_error = "no error";

cb_status fail(cb_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

cb_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CB_OK;
  return fail(CB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cb_status need_tensor(const void* p, const char* name) {
  if (p == nullptr) return fail(CB_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(CB_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return CB_OK;
}

cb_status need_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(CB_ERR_INVALID_ARG, "%s is NULL", name);
  return CB_OK;
}

#define CB_TRY(expr)                  \
  do {                                \
    const cb_status _s = (expr);      \
    if (_s != CB_OK) return _s;       \
  } while (0)

cb_status check_plan(const cb_plan* plan) {
  if (plan == nullptr) return fail(CB_ERR_INVALID_ARG, "plan is NULL");
  return CB_OK;
}

cb::RopeTable table(const cb_plan* p) { return cb::RopeTable{p->rope_tab, p->n_tokens}; }

int32_t k_for_ratio(int32_t r_pct, int32_t n_ctx) {
  return static_cast<int32_t>((static_cast<int64_t>(r_pct) * n_ctx) / 100);
}

}  // namespace

namespace cb {
cb_status set_last_error(cb_status s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace cb

extern "C" {

int32_t cb_version(void) { return 100; }

const char* cb_last_error_string(void) { return g_last_error.c_str(); }

cb_status cb_plan_create(const cb_config* cfg, cb_plan** out) {
  CB_NVTX_RANGE();
  CB_TRY(need_ptr(cfg, "cfg"));
  CB_TRY(need_ptr(out, "out"));
  *out = nullptr;
  const cb_config& c = *cfg;
  if (c.n_chunks < 0 || c.chunk_len <= 0 || c.n_suffix < 0)
    return fail(CB_ERR_INVALID_ARG, "n_chunks >= 0, chunk_len > 0 and n_suffix >= 0 required");
  const int64_t n_tokens = (int64_t)c.n_chunks * c.chunk_len + c.n_suffix;
  if (n_tokens <= 0 || n_tokens > (1 << 24)) return fail(CB_ERR_INVALID_ARG, "n_tokens must be in [1, 2^24]");
  if (c.hkv <= 0 || c.hq <= 0 || c.hq % c.hkv != 0)
    return fail(CB_ERR_INVALID_ARG, "hq must be a positive multiple of hkv");
  const int group = c.hq / c.hkv;
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16)
    return fail(CB_ERR_UNSUPPORTED, "hq / hkv = %d; supported: 1, 2, 4, 8, 16", group);
  if (c.head_dim != 64 && c.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "head_dim %d; supported: 64, 128", c.head_dim);
  if (c.hkv * c.head_dim > 2048) return fail(CB_ERR_UNSUPPORTED, "hkv * head_dim above 2048");
  if (!(c.rope_theta > 1.0) || !std::isfinite(c.rope_theta)) return fail(CB_ERR_INVALID_ARG, "rope_theta must be > 1");
  if (c.rope_style != CB_ROPE_HALF && c.rope_style != CB_ROPE_INTERLEAVED)
    return fail(CB_ERR_INVALID_ARG, "unknown rope_style %d", c.rope_style);
  if (c.r1_pct < 0 || c.r1_pct > 100 || c.r2_pct < 0 || c.r2_pct > c.r1_pct)
    return fail(CB_ERR_INVALID_ARG, "need 0 <= r2_pct <= r1_pct <= 100");
  if (c.deviation != CB_DEV_V && c.deviation != CB_DEV_KV)
    return fail(CB_ERR_INVALID_ARG, "unknown deviation %d", c.deviation);
  if (c.filter != CB_FILTER_KEEP && c.filter != CB_FILTER_RESELECT)
    return fail(CB_ERR_INVALID_ARG, "unknown filter %d", c.filter);

  cb_plan* p = new cb_plan();
  p->cfg = c;
  p->n_ctx = c.n_chunks * c.chunk_len;
  p->n_tokens = (int32_t)n_tokens;
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaMalloc(&p->rope_tab, sizeof(float2) * (size_t)n_tokens * (c.head_dim / 2));
  if (e == cudaSuccess) e = cudaMalloc(&p->err, 2 * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->aux_stream, cudaStreamNonBlocking);
  for (int a = 1; a < kAttnStreams && e == cudaSuccess; ++a)
    e = cudaStreamCreateWithFlags(&p->aux_attn[a], cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming);
  if (e == cudaSuccess) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    p->decode.sms = sms > 0 ? sms : 1;
  }
  const size_t dec_units = (size_t)c.hq * cb::decode_max_splits();  // (kv head, split, q head) triples
  if (e == cudaSuccess) e = cudaMalloc(&p->decode.part_o, sizeof(float) * dec_units * c.head_dim);
  if (e == cudaSuccess) e = cudaMalloc(&p->decode.part_ml, sizeof(float2) * dec_units);
  if (e == cudaSuccess) e = cudaMalloc(&p->decode.tickets, sizeof(int32_t) * c.hkv);
  if (e == cudaSuccess) e = cudaMemset(p->decode.tickets, 0, sizeof(int32_t) * c.hkv);

  if (e == cudaSuccess) {
    const int32_t init[2] = {0, -1};
    e = cudaMemcpy(p->err, init, sizeof(init), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    // (cos, sin) of p * theta^(-2j/D): the exponent (-2j)/D, theta^x, the angle and cos / sin in
    // fp64 with the C library's routines, then rounded to fp32.
    const int half = c.head_dim / 2;
    std::vector<double> inv(half);
    for (int j = 0; j < half; ++j) inv[j] = std::pow(c.rope_theta, (-2.0 * j) / c.head_dim);
    std::vector<float2> tab((size_t)n_tokens * half);
    for (int64_t pos = 0; pos < n_tokens; ++pos)
      for (int j = 0; j < half; ++j) {
        const double a = (double)pos * inv[j];
        tab[(size_t)pos * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    e = cudaMemcpy(p->rope_tab, tab.data(), sizeof(float2) * tab.size(), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cb_plan_destroy(p);
    return cuda_status(e, "cb_plan_create");
  }
  *out = p;
  return CB_OK;
}

cb_status cb_plan_destroy(cb_plan* plan) {
  CB_NVTX_RANGE();
  if (plan == nullptr) return CB_OK;
  cudaDeviceSynchronize();
  cudaFree(plan->rope_tab);
  cudaFree(plan->err);
  cudaFree(plan->decode.part_o);
  cudaFree(plan->decode.part_ml);
  cudaFree(plan->decode.tickets);
  if (plan->aux_stream) cudaStreamDestroy(plan->aux_stream);
  for (int a = 1; a < kAttnStreams; ++a)
    if (plan->aux_attn[a]) cudaStreamDestroy(plan->aux_attn[a]);
  if (plan->ev_fork) cudaEventDestroy(plan->ev_fork);
  if (plan->ev_ready) cudaEventDestroy(plan->ev_ready);
  if (plan->ev_join) cudaEventDestroy(plan->ev_join);
  delete plan;
  return CB_OK;
}

cb_status cb_layer_sizes(const cb_plan* plan, int32_t layer, int32_t* n_cand, int32_t* k, int32_t* mq,
                         int32_t* selects) {
  CB_TRY(check_plan(plan));
  if (layer < 1) return fail(CB_ERR_INVALID_ARG, "layer is 1-based, got %d", layer);
  const int32_t k1 = k_for_ratio(plan->cfg.r1_pct, plan->n_ctx);
  const int32_t k2 = k_for_ratio(plan->cfg.r2_pct, plan->n_ctx);
  int32_t c, kk, sel;
  if (layer == 1) {
    c = plan->n_ctx, kk = k1, sel = 1;
  } else if (layer == 2) {
    c = k1, kk = k2, sel = 1;
  } else if (plan->cfg.filter == CB_FILTER_RESELECT) {
    c = k1, kk = k2, sel = 1;
  } else {
    c = k2, kk = k2, sel = 0;
  }
  if (n_cand) *n_cand = c;
  if (k) *k = kk;
  if (mq) *mq = kk + plan->cfg.n_suffix;
  if (selects) *selects = sel;
  return CB_OK;
}

cb_status cb_rope_rerotate(cb_plan* plan, void* out, const void* x, const int32_t* in_rows,
                           const int32_t* out_rows, const int32_t* pos_from, const int32_t* pos_to, int32_t n,
                           int32_t n_heads, int32_t x_rows, int32_t out_rows_total, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (n < 0 || n_heads <= 0 || x_rows < 0 || out_rows_total < 0)
    return fail(CB_ERR_INVALID_ARG, "negative size or n_heads <= 0");
  if (n == 0) return CB_OK;
  CB_TRY(need_tensor(out, "out"));
  CB_TRY(need_tensor(x, "x"));
  CB_TRY(need_ptr(pos_to, "pos_to"));
  if (out == x && (in_rows != nullptr || out_rows != nullptr))
    return fail(CB_ERR_INVALID_ARG, "in-place rotation needs in_rows == out_rows == NULL");
  const cb::RowMap im{in_rows, n, 0, x_rows};
  const cb::RowMap om{out_rows, n, 0, out_rows_total};
  return cuda_status(cb::launch_rope_rows(out, x, im, om, pos_from, pos_to, nullptr, n, n_heads,
                                          plan->cfg.head_dim, plan->cfg.rope_style, table(plan), plan->err,
                                          static_cast<cudaStream_t>(stream)),
                     "cb_rope_rerotate");
}

cb_status cb_kv_deviation(cb_plan* plan, const void* v_new, const void* v_old, const int32_t* cand, int32_t m,
                          float* dev, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (m < 0) return fail(CB_ERR_INVALID_ARG, "m < 0");
  if (m == 0) return CB_OK;
  if (cand == nullptr && m > plan->n_ctx) return fail(CB_ERR_INVALID_ARG, "m > n_ctx without a candidate list");
  CB_TRY(need_tensor(v_new, "v_new"));
  CB_TRY(need_tensor(v_old, "v_old"));
  CB_TRY(need_ptr(dev, "dev"));
  return cuda_status(cb::launch_kv_deviation(nullptr, nullptr, v_new, v_old, cand, m, plan->n_ctx, plan->cfg.hkv,
                                             plan->cfg.head_dim, 1, 0, table(plan), dev, plan->err,
                                             static_cast<cudaStream_t>(stream)),
                     "cb_kv_deviation");
}

cb_status cb_kv_deviation_kv(cb_plan* plan, const void* k_new, const void* k_old, const void* v_new,
                             const void* v_old, const int32_t* cand, int32_t m, float* dev, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (m < 0) return fail(CB_ERR_INVALID_ARG, "m < 0");
  if (m == 0) return CB_OK;
  if (cand == nullptr && m > plan->n_ctx) return fail(CB_ERR_INVALID_ARG, "m > n_ctx without a candidate list");
  CB_TRY(need_tensor(k_new, "k_new"));
  CB_TRY(need_tensor(k_old, "k_old"));
  CB_TRY(need_tensor(v_new, "v_new"));
  CB_TRY(need_tensor(v_old, "v_old"));
  CB_TRY(need_ptr(dev, "dev"));
  const auto& c = plan->cfg;
  return cuda_status(cb::launch_kv_deviation(k_new, k_old, v_new, v_old, cand, m, plan->n_ctx, c.hkv, c.head_dim,
                                             c.chunk_len, c.rope_style, table(plan), dev, plan->err,
                                             static_cast<cudaStream_t>(stream)),
                     "cb_kv_deviation_kv");
}

cb_status cb_hkvd_topk(cb_plan* plan, const float* dev, const int32_t* cand, int32_t m, int32_t k,
                       int32_t* sel_tok, int32_t* sel_row, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (m < 0 || k < 0 || k > m) return fail(CB_ERR_INVALID_ARG, "need 0 <= k <= m (k=%d, m=%d)", k, m);
  if (k == 0) return CB_OK;
  CB_TRY(need_ptr(dev, "dev"));
  CB_TRY(need_ptr(sel_tok, "sel_tok"));
  CB_TRY(need_ptr(sel_row, "sel_row"));
  return cuda_status(cb::launch_hkvd_topk(dev, cand, m, k, sel_tok, sel_row, plan->err,
                                          static_cast<cudaStream_t>(stream)),
                     "cb_hkvd_topk");
}

cb_status cb_fuse_scatter(cb_plan* plan, void* k_fused, void* v_fused, const void* k_new, const void* v_new,
                          const int32_t* sel_tok, int32_t k, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (k < 0 || k > plan->n_ctx) return fail(CB_ERR_INVALID_ARG, "need 0 <= k <= n_ctx");
  if (k + plan->cfg.n_suffix == 0) return CB_OK;
  CB_TRY(need_tensor(k_fused, "k_fused"));
  CB_TRY(need_tensor(v_fused, "v_fused"));
  CB_TRY(need_tensor(k_new, "k_new"));
  CB_TRY(need_tensor(v_new, "v_new"));
  if (k > 0) CB_TRY(need_ptr(sel_tok, "sel_tok"));
  return cuda_status(cb::launch_fuse_scatter(k_fused, v_fused, k_new, v_new, sel_tok, k, plan->n_ctx,
                                             plan->n_tokens, plan->cfg.hkv, plan->cfg.head_dim,
                                             plan->cfg.rope_style, table(plan), plan->err,
                                             static_cast<cudaStream_t>(stream)),
                     "cb_fuse_scatter");
}

cb_status cb_hkvd_attention(cb_plan* plan, const void* q, const int32_t* q_pos, int32_t mq, const void* k,
                            const void* v, int32_t n_keys, float scale, void* out, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (mq < 0 || n_keys < 0) return fail(CB_ERR_INVALID_ARG, "negative size");
  if (mq == 0) return CB_OK;
  if (n_keys == 0) return fail(CB_ERR_INVALID_ARG, "n_keys == 0 with queries to answer");
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_ptr(q_pos, "q_pos"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  CB_TRY(need_tensor(out, "out"));
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt((float)plan->cfg.head_dim);
  const cb::QueryPositions qp{q_pos, mq, 0, true};
  return cuda_status(cb::launch_hkvd_attention(q, qp, mq, k, v, n_keys, plan->cfg.hq, plan->cfg.hkv,
                                               plan->cfg.head_dim, scale, out, plan->err,
                                               static_cast<cudaStream_t>(stream)),
                     "cb_hkvd_attention");
}

int32_t cb_attention_uses_paired_tiles(const cb_plan* plan, int32_t mq) {
  if (plan == nullptr) return 0;
  return cb::attention_pp_eligible(mq, plan->cfg.hq, plan->cfg.hkv, plan->cfg.head_dim) ? 1 : 0;
}

cb_status cb_test_attention_wait_timeout(cb_plan* plan, const void* q, const int32_t* q_pos, int32_t mq,
                                         const void* k, const void* v, int32_t n_keys, void* out, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (plan->cfg.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "the wait-timeout probe needs head_dim 128");
  if (mq <= 0 || n_keys <= 128) return fail(CB_ERR_INVALID_ARG, "the wait-timeout probe needs mq > 0, n_keys > 128");
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_ptr(q_pos, "q_pos"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  CB_TRY(need_tensor(out, "out"));
  const cb::QueryPositions qp{q_pos, mq, 0, true};
  return cuda_status(cb::launch_attention_timeout_probe(q, qp, mq, k, v, n_keys, plan->cfg.hq, plan->cfg.hkv,
                                                        1.0f / std::sqrt(128.0f), out, plan->err,
                                                        static_cast<cudaStream_t>(stream)),
                     "cb_test_attention_wait_timeout");
}

cb_status cb_test_decode_wait_timeout(cb_plan* plan, const void* q, const void* k, const void* v, int32_t n_keys,
                                      void* out, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (plan->cfg.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "the wait-timeout probe needs head_dim 128");
  if (n_keys <= 128) return fail(CB_ERR_INVALID_ARG, "the wait-timeout probe needs n_keys > 128");
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  CB_TRY(need_tensor(out, "out"));
  const auto& c = plan->cfg;
  return cuda_status(cb::launch_decode_timeout_probe(q, k, v, n_keys, c.hq, c.hkv, 1.0f / std::sqrt(128.0f), out,
                                                     plan->decode, plan->err, static_cast<cudaStream_t>(stream)),
                     "cb_test_decode_wait_timeout");
}

cb_status cb_test_projection_wait_timeout(cb_plan* plan, const void* x, int32_t d_model, int32_t m,
                                          const void* w_qkv, void* q, void* k, void* v, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (plan->cfg.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "the wait-timeout probe needs head_dim 128");
  if (m <= 0 || m > plan->n_tokens) return fail(CB_ERR_INVALID_ARG, "the wait-timeout probe needs 0 < m <= n_tokens");
  if (d_model < 128 || d_model % 64 != 0)
    return fail(CB_ERR_INVALID_ARG, "the wait-timeout probe needs d_model >= 128, a multiple of 64");
  CB_TRY(need_tensor(x, "x"));
  CB_TRY(need_tensor(w_qkv, "w_qkv"));
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  const auto& c = plan->cfg;
  return cuda_status(cb::launch_projection_timeout_probe(x, d_model, m, w_qkv, plan->n_tokens, c.hq, c.hkv, q, k, v,
                                                         plan->err, static_cast<cudaStream_t>(stream)),
                     "cb_test_projection_wait_timeout");
}

cb_status cb_attention_sparsity(cb_plan* plan, const void* q, const int32_t* q_pos, int32_t mq, const void* k,
                                const void* v, int32_t n_keys, float scale, float eps, void* out, void* row_stats,
                                int32_t* counts, uint64_t* total, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (mq < 0 || n_keys < 0) return fail(CB_ERR_INVALID_ARG, "negative size");
  if (!(eps > 0.0f) || !std::isfinite(eps)) return fail(CB_ERR_INVALID_ARG, "eps must be positive and finite");
  CB_TRY(need_ptr(total, "total"));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mq == 0) return cuda_status(cudaMemsetAsync(total, 0, sizeof(uint64_t), s), "cb_attention_sparsity");
  if (n_keys == 0) return fail(CB_ERR_INVALID_ARG, "n_keys == 0 with queries to answer");
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_ptr(q_pos, "q_pos"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  CB_TRY(need_tensor(out, "out"));
  CB_TRY(need_tensor(row_stats, "row_stats"));
  CB_TRY(need_ptr(counts, "counts"));
  const auto& c = plan->cfg;
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt((float)c.head_dim);
  const cb::QueryPositions qp{q_pos, mq, 0, true};
  cb::AttentionDiag first;  // pass 1: the attention and each row's (max, sum)
  first.row_stats = static_cast<float2*>(row_stats);
  CB_TRY(cuda_status(cb::launch_hkvd_attention(q, qp, mq, k, v, n_keys, c.hq, c.hkv, c.head_dim, scale, out, plan->err,
                                               s, first),
                     "cb_attention_sparsity (statistics pass)"));
  cb::AttentionDiag second;  // pass 2: the same scores against each row's threshold
  second.count_stats = static_cast<const float2*>(row_stats);
  second.log2_eps = std::log2(eps);
  second.counts = counts;
  CB_TRY(cuda_status(cb::launch_hkvd_attention(q, qp, mq, k, v, n_keys, c.hq, c.hkv, c.head_dim, scale, out, plan->err,
                                               s, second),
                     "cb_attention_sparsity (counting pass)"));
  return cuda_status(cb::launch_sum_counts(counts, (int64_t)mq * c.hq, reinterpret_cast<unsigned long long*>(total), s),
                     "cb_attention_sparsity (sum)");
}

cb_status cb_output_deviation(cb_plan* plan, const void* o, const void* o_ref, int32_t rows, double* sums,
                              void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (rows < 0) return fail(CB_ERR_INVALID_ARG, "rows < 0");
  CB_TRY(need_ptr(sums, "sums"));
  if (rows > 0) {
    CB_TRY(need_tensor(o, "o"));
    CB_TRY(need_tensor(o_ref, "o_ref"));
  }
  const int64_t n = (int64_t)rows * plan->cfg.hq * plan->cfg.head_dim;
  return cuda_status(cb::launch_output_deviation(o, o_ref, n, sums, static_cast<cudaStream_t>(stream)),
                     "cb_output_deviation");
}

static cb_status qkv_projection(const char* fn, cb_plan* plan, const void* x, int32_t x_rows, int32_t d_model,
                                const int32_t* x_index, const int32_t* tokens, int32_t m, const void* w_qkv,
                                int32_t encode, void* x_gathered, void* q, void* k, void* v, void* stream) {
  CB_TRY(check_plan(plan));
  if (m < 0 || x_rows < 0) return fail(CB_ERR_INVALID_ARG, "negative size");
  if (m == 0) return CB_OK;
  if (!cb::qkv_projection_supported(d_model))
    return fail(CB_ERR_UNSUPPORTED, "d_model %d: a positive multiple of 64 is required", d_model);
  if (x_index == nullptr && m > x_rows) return fail(CB_ERR_INVALID_ARG, "m > x_rows without an index list");
  if (tokens == nullptr && m > plan->n_tokens) return fail(CB_ERR_INVALID_ARG, "m > n_tokens without a token list");
  CB_TRY(need_tensor(x, "x"));
  CB_TRY(need_tensor(w_qkv, "w_qkv"));
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  if (x_index != nullptr) CB_TRY(need_tensor(x_gathered, "x_gathered"));
  const auto& c = plan->cfg;
  return cuda_status(cb::launch_qkv_projection(x, x_rows, d_model, x_index, tokens, m, x_gathered, w_qkv,
                                               plan->n_tokens, c.hq, c.hkv, c.head_dim, encode ? 1 : 0, c.rope_style,
                                               table(plan), q, k, v, plan->err, static_cast<cudaStream_t>(stream)),
                     fn);
}

cb_status cb_qkv_projection(cb_plan* plan, const void* x, int32_t x_rows, int32_t d_model, const int32_t* rows,
                            int32_t m, const void* w_qkv, int32_t encode, void* x_gathered, void* q, void* k, void* v,
                            void* stream) {
  CB_NVTX_RANGE();
  return qkv_projection("cb_qkv_projection", plan, x, x_rows, d_model, rows, rows, m, w_qkv, encode, x_gathered, q,
                        k, v, stream);
}

cb_status cb_qkv_projection_indexed(cb_plan* plan, const void* x, int32_t x_rows, int32_t d_model,
                                    const int32_t* x_index, const int32_t* tokens, int32_t m, const void* w_qkv,
                                    int32_t encode, void* x_gathered, void* q, void* k, void* v, void* stream) {
  CB_NVTX_RANGE();
  return qkv_projection("cb_qkv_projection_indexed", plan, x, x_rows, d_model, x_index, tokens, m, w_qkv, encode,
                        x_gathered, q, k, v, stream);
}

cb_status cb_decode_attention(cb_plan* plan, const void* q, const void* k, const void* v, int32_t n_keys,
                              float scale, void* out, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (n_keys < 0) return fail(CB_ERR_INVALID_ARG, "n_keys < 0");
  if (n_keys == 0) return CB_OK;
  CB_TRY(need_tensor(q, "q"));
  CB_TRY(need_tensor(k, "k"));
  CB_TRY(need_tensor(v, "v"));
  CB_TRY(need_tensor(out, "out"));
  const auto& c = plan->cfg;
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt((float)c.head_dim);
  if (!cb::decode_tc_supported(c.hq, c.hkv, c.head_dim))
    return fail(CB_ERR_UNSUPPORTED, "decode: hq / hkv = %d, head_dim %d", c.hq / c.hkv, c.head_dim);
  return cuda_status(cb::launch_decode_tc(q, k, v, n_keys, c.hq, c.hkv, c.head_dim, scale, out, plan->decode,
                                          plan->err, static_cast<cudaStream_t>(stream)),
                     "cb_decode_attention");
}

struct LayerShape {
  int32_t n_cand, k, mq, selects;
};

// Host checks of one layer's buffers; `cand` is the candidate list the layer will read.
static cb_status validate_io(cb_plan* plan, int32_t layer, const cb_layer_io* io, const int32_t* cand,
                             LayerShape* sh) {
  CB_TRY(need_ptr(io, "io"));
  CB_TRY(cb_layer_sizes(plan, layer, &sh->n_cand, &sh->k, &sh->mq, &sh->selects));
  CB_TRY(need_tensor(io->k_old, "io.k_old"));
  CB_TRY(need_tensor(io->v_old, "io.v_old"));
  CB_TRY(need_tensor(io->k_new, "io.k_new"));
  CB_TRY(need_tensor(io->v_new, "io.v_new"));
  CB_TRY(need_tensor(io->q, "io.q"));
  CB_TRY(need_tensor(io->k_fused, "io.k_fused"));
  CB_TRY(need_tensor(io->v_fused, "io.v_fused"));
  if (sh->mq > 0) {
    CB_TRY(need_tensor(io->q_rot, "io.q_rot"));
    CB_TRY(need_tensor(io->out, "io.out"));
  }
  if (sh->k > 0) {
    CB_TRY(need_ptr(io->sel_tok, "io.sel_tok"));
    CB_TRY(need_ptr(io->sel_row, "io.sel_row"));
  }
  if (layer >= 2 && sh->n_cand > 0) CB_TRY(need_ptr(cand, "io.cand"));
  if (sh->selects && sh->n_cand > 0) CB_TRY(need_ptr(io->dev, "io.dev"));
  return CB_OK;
}

// One stage of layer `layer` on `s`; `cand` is the candidate list the layer reads (ignored at
// layer 1, where the candidates are all context tokens). S_l is sel_tok at selecting layers and
// the candidates themselves elsewhere; the fuse pass then copies them out to sel_tok / sel_row.
// inputs_by_event: the attention's inputs are ordered by an event on its stream (cb_blend_request),
// so it need not wait for the kernel before it on that stream, which it does not read from.
static cb_status enqueue_stage(cb_plan* plan, int32_t layer, const cb_layer_io* io, const int32_t* cand,
                               const LayerShape& sh, int32_t stage, cudaStream_t s, bool inputs_by_event = false) {
  const auto& c = plan->cfg;
  if (layer == 1) cand = nullptr;
  const int32_t* sel = sh.selects ? io->sel_tok : cand;
  switch (stage) {
    case CB_STAGE_DEVIATION: {
      if (!sh.selects) return CB_OK;
      const bool kv = c.deviation == CB_DEV_KV;
      return cuda_status(cb::launch_kv_deviation(kv ? io->k_new : nullptr, kv ? io->k_old : nullptr, io->v_new,
                                                 io->v_old, cand, sh.n_cand, plan->n_ctx, c.hkv, c.head_dim,
                                                 c.chunk_len, c.rope_style, table(plan), io->dev, plan->err, s),
                         "deviation");
    }
    case CB_STAGE_TOPK:
      if (!sh.selects) return CB_OK;
      return cuda_status(cb::launch_hkvd_topk(io->dev, cand, sh.n_cand, sh.k, io->sel_tok, io->sel_row, plan->err, s),
                         "top-k");
    case CB_STAGE_FUSE: {
      // One launch: the fused cache and the query encoding (both read the layer's selection list).
      // Small blocks on the layers whose attention runs the paired-tile kernel (see the fuse kernel).
      const bool copy_out = !sh.selects && sh.k > 0;
      const bool narrow = cb::attention_pp_eligible(sh.mq, c.hq, c.hkv, c.head_dim);
      return cuda_status(cb::launch_blend_fuse(io->k_fused, io->v_fused, io->k_old, io->v_old, io->k_new, io->v_new,
                                               sel, sh.k, copy_out ? io->sel_tok : nullptr,
                                               copy_out ? io->sel_row : nullptr, plan->n_ctx, c.chunk_len,
                                               plan->n_tokens, c.hkv, c.head_dim, c.rope_style, table(plan),
                                               sh.mq > 0 ? io->q : nullptr, sh.mq > 0 ? io->q_rot : nullptr, sh.mq,
                                               c.hq, narrow, plan->err, s),
                         "fuse");
    }
    case CB_STAGE_ATTENTION: {
      if (sh.mq == 0) return CB_OK;
      // query row t sits at sel[t] (t < k) or n_ctx + t - k
      const cb::QueryPositions qp{sel, sh.k, plan->n_ctx, !inputs_by_event};
      return cuda_status(cb::launch_hkvd_attention(io->q_rot, qp, sh.mq, io->k_fused, io->v_fused, plan->n_tokens,
                                                   c.hq, c.hkv, c.head_dim, 1.0f / std::sqrt((float)c.head_dim),
                                                   io->out, plan->err, s),
                         "attention");
    }
    default:
      return fail(CB_ERR_INVALID_ARG, "unknown stage %d", stage);
  }
}

// The selections of layers 2..n_layers (all from cand = S_1, k_2 each), kSelectBatchMax layers per
// pair of launches.
static cb_status enqueue_select_batches(cb_plan* plan, int32_t n_layers, const cb_layer_io* ios,
                                        const int32_t* cand, const LayerShape& sh, cudaStream_t s) {
  const auto& c = plan->cfg;
  const bool kv = c.deviation == CB_DEV_KV;
  for (int32_t l0 = 2; l0 <= n_layers; l0 += cb::kSelectBatchMax) {
    cb::SelectBatch b = {};
    b.n = std::min<int32_t>(cb::kSelectBatchMax, n_layers - l0 + 1);
    for (int i = 0; i < b.n; ++i) {
      const cb_layer_io& io = ios[l0 - 1 + i];
      b.k_new[i] = kv ? io.k_new : nullptr;
      b.k_old[i] = kv ? io.k_old : nullptr;
      b.v_new[i] = io.v_new;
      b.v_old[i] = io.v_old;
      b.dev[i] = io.dev;
      b.sel_tok[i] = io.sel_tok;
      b.sel_row[i] = io.sel_row;
    }
    CB_TRY(cuda_status(cb::launch_select_batch(b, cand, sh.n_cand, sh.k, plan->n_ctx, c.hkv, c.head_dim, c.chunk_len,
                                               c.rope_style, table(plan), plan->err, s),
                       "batched selection"));
  }
  return CB_OK;
}

cb_status cb_blend_layer(cb_plan* plan, int32_t layer, const cb_layer_io* io, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  LayerShape sh;
  CB_TRY(validate_io(plan, layer, io, io ? io->cand : nullptr, &sh));
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t st = CB_STAGE_DEVIATION; st <= CB_STAGE_ATTENTION; ++st)
    CB_TRY(enqueue_stage(plan, layer, io, io->cand, sh, st, s));
  return CB_OK;
}

cb_status cb_blend_stage(cb_plan* plan, int32_t layer, const cb_layer_io* io, int32_t stage, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (stage < CB_STAGE_DEVIATION || stage > CB_STAGE_ATTENTION) return fail(CB_ERR_INVALID_ARG, "unknown stage %d", stage);
  LayerShape sh;
  CB_TRY(validate_io(plan, layer, io, io ? io->cand : nullptr, &sh));
  return enqueue_stage(plan, layer, io, io->cand, sh, stage, static_cast<cudaStream_t>(stream));
}

cb_status cb_blend_request(cb_plan* plan, int32_t n_layers, const cb_layer_io* ios, void* stream) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  if (n_layers < 1) return fail(CB_ERR_INVALID_ARG, "n_layers must be >= 1");
  CB_TRY(need_ptr(ios, "ios"));
  // C_l is the selection of layer l - 1, or of layer 1 when every layer re-selects from its pool.
  const bool reselect = plan->cfg.filter == CB_FILTER_RESELECT;
  auto cand_of = [&](int32_t l) -> const int32_t* {
    return l == 1 ? nullptr : ios[(reselect ? 1 : l - 1) - 1].sel_tok;
  };
  for (int32_t l = 1; l <= n_layers; ++l) {
    LayerShape sh;
    CB_TRY(validate_io(plan, l, &ios[l - 1], cand_of(l), &sh));
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t attn_stream[kAttnStreams];
  attn_stream[0] = s;
  for (int a = 1; a < kAttnStreams; ++a) attn_stream[a] = plan->aux_attn[a];
  CB_TRY(cuda_status(cudaEventRecord(plan->ev_fork, s), "fork"));
  CB_TRY(cuda_status(cudaStreamWaitEvent(plan->aux_stream, plan->ev_fork, 0), "fork"));
  for (int a = 1; a < kAttnStreams; ++a)
    CB_TRY(cuda_status(cudaStreamWaitEvent(attn_stream[a], plan->ev_fork, 0), "fork"));
  // Re-selection: every layer >= 2 selects k_2 from the same candidates S_1, so their deviations and
  // top-k go out as two batched launches right after layer 1's selection (instead of a deviation and
  // a one-block top-k ahead of every fuse), and the fuses then run ahead of the attention as they do
  // when the set is kept.
  const bool batch_select = reselect && n_layers >= 2;
  for (int32_t l = 1; l <= n_layers; ++l) {
    const cb_layer_io* io = &ios[l - 1];
    const int32_t* cand = cand_of(l);
    LayerShape sh;
    CB_TRY(validate_io(plan, l, io, cand, &sh));
    if (batch_select && l >= 2) {
      if (l == 2) CB_TRY(enqueue_select_batches(plan, n_layers, ios, ios[0].sel_tok, sh, plan->aux_stream));
      CB_TRY(enqueue_stage(plan, l, io, cand, sh, CB_STAGE_FUSE, plan->aux_stream));
    } else {
      for (int32_t st = CB_STAGE_DEVIATION; st <= CB_STAGE_FUSE; ++st)
        CB_TRY(enqueue_stage(plan, l, io, cand, sh, st, plan->aux_stream));
    }
    const cudaStream_t a = attn_stream[(l - 1) % kAttnStreams];
    CB_TRY(cuda_status(cudaEventRecord(plan->ev_ready, plan->aux_stream), "layer inputs ready"));
    CB_TRY(cuda_status(cudaStreamWaitEvent(a, plan->ev_ready, 0), "layer inputs ready"));
    CB_TRY(enqueue_stage(plan, l, io, cand, sh, CB_STAGE_ATTENTION, a, true));
  }
  for (int a = 1; a < kAttnStreams; ++a) {
    CB_TRY(cuda_status(cudaEventRecord(plan->ev_join, attn_stream[a]), "join"));
    CB_TRY(cuda_status(cudaStreamWaitEvent(s, plan->ev_join, 0), "join"));
  }
  CB_TRY(cuda_status(cudaEventRecord(plan->ev_join, plan->aux_stream), "join"));
  return cuda_status(cudaStreamWaitEvent(s, plan->ev_join, 0), "join");
}

cb_status cb_check(cb_plan* plan) {
  CB_NVTX_RANGE();
  CB_TRY(check_plan(plan));
  int32_t h[2] = {0, -1};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(h, plan->err, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) {
    const int32_t init[2] = {0, -1};
    e = cudaMemcpy(plan->err, init, sizeof(init), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) return cuda_status(e, "cb_check");
  if (h[0] == 0) return CB_OK;
  const bool timeout = (h[0] & cb::kErrTimeout) != 0;
  return fail(timeout ? CB_ERR_TIMEOUT : CB_ERR_DEVICE_CHECK,
              "device check failed: flags 0x%x (1 rope range, 2 index, 4 order, 8 timeout), first at %d", h[0], h[1]);
}

}  // extern "C"
