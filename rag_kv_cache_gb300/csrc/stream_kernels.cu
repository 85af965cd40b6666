// HBM-streaming kernels of the blend: RoPE table, row rotation (re-rotation
// of cached keys and encoding of recomputed rows), V deviation, fused-cache
// construction and scatter, and the single-block HKVD top-k.
//
// Sources: "数学推导" §RoPE 位置编码的相对位置不变性证明 (pair rotation),
// §CacheBlend 中的应用 (k_new = R_{p_new - p_old} k_old), §形式化 (fused KV),
// §近似解 (TopK of ||V_new - V_old||^2); "rag的kvcache问题" §渐进式过滤机制.
#include "common.cuh"
#include "kernels.h"

namespace cb {

namespace {

constexpr int kWarp = 32;

__device__ __forceinline__ int map_row(const RowMap& m, int i) {
  return i < m.k ? (m.idx ? m.idx[i] : i) : m.base + (i - m.k);
}

// Rotate one row of n_heads x D bf16 by the table row `cs` (sign of sin flipped when neg).
// One warp per row; 16-byte accesses; src may equal dst.
template <int STYLE, int B>
__device__ __forceinline__ void rotate_row(uint8_t* dst, const uint8_t* src, int n_heads, int head_dim,
                                           const float2* __restrict__ cs, bool neg, int lane) {
  if (STYLE == 0) {
    // pair (j, j + D/2): a unit is 8 consecutive j of one head, lo and hi halves.
    const int per_head = head_dim / 16;
    const int units = n_heads * per_head;
    const int half_bytes = head_dim;  // D/2 elements * 2 bytes
    for (int u0 = lane; u0 < units; u0 += kWarp * B) {
      uint4 lo[B], hi[B];
#pragma unroll
      for (int q = 0; q < B; ++q) {
        const int u = u0 + kWarp * q;
        if (u < units) {
          const int h = u / per_head, c = u % per_head;
          const uint8_t* p = src + (size_t)h * head_dim * 2 + c * 16;
          lo[q] = ld_stream(p);
          hi[q] = ld_stream(p + half_bytes);
        }
      }
#pragma unroll
      for (int q = 0; q < B; ++q) {
        const int u = u0 + kWarp * q;
        if (u < units) {
          const int h = u / per_head, c = u % per_head;
          float a[8], b[8], oa[8], ob[8];
          unpack8(lo[q], a);
          unpack8(hi[q], b);
          const float4* t4 = reinterpret_cast<const float4*>(cs + c * 8);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 t = __ldg(t4 + e);
            const float c0 = t.x, s0 = neg ? -t.y : t.y, c1 = t.z, s1 = neg ? -t.w : t.w;
            oa[2 * e] = a[2 * e] * c0 - b[2 * e] * s0;
            ob[2 * e] = a[2 * e] * s0 + b[2 * e] * c0;
            oa[2 * e + 1] = a[2 * e + 1] * c1 - b[2 * e + 1] * s1;
            ob[2 * e + 1] = a[2 * e + 1] * s1 + b[2 * e + 1] * c1;
          }
          uint8_t* p = dst + (size_t)h * head_dim * 2 + c * 16;
          st_stream(p, pack8(oa));
          st_stream(p + half_bytes, pack8(ob));
        }
      }
    }
  } else {
    // pair (2j, 2j + 1): a unit is one 16-byte vector = 4 pairs.
    const int per_head = head_dim / 8;
    const int units = n_heads * per_head;
    for (int u0 = lane; u0 < units; u0 += kWarp * B) {
      uint4 v[B];
#pragma unroll
      for (int q = 0; q < B; ++q) {
        const int u = u0 + kWarp * q;
        if (u < units) v[q] = ld_stream(src + (size_t)u * 16);
      }
#pragma unroll
      for (int q = 0; q < B; ++q) {
        const int u = u0 + kWarp * q;
        if (u < units) {
          const int c = u % per_head;
          float a[8], o[8];
          unpack8(v[q], a);
          const float4* t4 = reinterpret_cast<const float4*>(cs + c * 4);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float4 t = __ldg(t4 + e);
            const float c0 = t.x, s0 = neg ? -t.y : t.y, c1 = t.z, s1 = neg ? -t.w : t.w;
            o[4 * e + 0] = a[4 * e + 0] * c0 - a[4 * e + 1] * s0;
            o[4 * e + 1] = a[4 * e + 0] * s0 + a[4 * e + 1] * c0;
            o[4 * e + 2] = a[4 * e + 2] * c1 - a[4 * e + 3] * s1;
            o[4 * e + 3] = a[4 * e + 2] * s1 + a[4 * e + 3] * c1;
          }
          st_stream(dst + (size_t)u * 16, pack8(o));
        }
      }
    }
  }
}

// Copy one row of `bytes` (multiple of 16) with a warp.
__device__ __forceinline__ void copy_row(uint8_t* dst, const uint8_t* src, int bytes, int lane) {
  constexpr int B = 4;
  const int vecs = bytes / 16;
  for (int u0 = lane; u0 < vecs; u0 += kWarp * B) {
    uint4 v[B];
#pragma unroll
    for (int q = 0; q < B; ++q)
      if (u0 + kWarp * q < vecs) v[q] = ld_stream(src + (size_t)(u0 + kWarp * q) * 16);
#pragma unroll
    for (int q = 0; q < B; ++q)
      if (u0 + kWarp * q < vecs) st_stream(dst + (size_t)(u0 + kWarp * q) * 16, v[q]);
  }
}

// Rotate pair-unit u of a row (half style: 8 frequencies of one head, lo and hi
// halves; interleaved: one 16-byte vector = 4 pairs).
template <int STYLE>
__device__ __forceinline__ void rotate_unit(uint8_t* dst, const uint8_t* src, int u, int head_dim,
                                            const float2* __restrict__ cs, bool neg) {
  if (STYLE == 0) {
    const int per_head = head_dim / 16;
    const int h = u / per_head, c = u % per_head;
    const size_t off = (size_t)h * head_dim * 2 + c * 16;
    const uint4 lo = ld_stream(src + off), hi = ld_stream(src + off + head_dim);
    float a[8], b[8], oa[8], ob[8];
    unpack8(lo, a);
    unpack8(hi, b);
    const float4* t4 = reinterpret_cast<const float4*>(cs + c * 8);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 t = __ldg(t4 + e);
      const float c0 = t.x, s0 = neg ? -t.y : t.y, c1 = t.z, s1 = neg ? -t.w : t.w;
      oa[2 * e] = a[2 * e] * c0 - b[2 * e] * s0;
      ob[2 * e] = a[2 * e] * s0 + b[2 * e] * c0;
      oa[2 * e + 1] = a[2 * e + 1] * c1 - b[2 * e + 1] * s1;
      ob[2 * e + 1] = a[2 * e + 1] * s1 + b[2 * e + 1] * c1;
    }
    st_stream(dst + off, pack8(oa));
    st_stream(dst + off + head_dim, pack8(ob));
  } else {
    const int c = u % (head_dim / 8);
    const uint4 v = ld_stream(src + (size_t)u * 16);
    float a[8], o[8];
    unpack8(v, a);
    const float4* t4 = reinterpret_cast<const float4*>(cs + c * 4);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float4 t = __ldg(t4 + e);
      const float c0 = t.x, s0 = neg ? -t.y : t.y, c1 = t.z, s1 = neg ? -t.w : t.w;
      o[4 * e + 0] = a[4 * e + 0] * c0 - a[4 * e + 1] * s0;
      o[4 * e + 1] = a[4 * e + 0] * s0 + a[4 * e + 1] * c0;
      o[4 * e + 2] = a[4 * e + 2] * c1 - a[4 * e + 3] * s1;
      o[4 * e + 3] = a[4 * e + 2] * s1 + a[4 * e + 3] * c1;
    }
    st_stream(dst + (size_t)u * 16, pack8(o));
  }
}

// One warp per (row, group of 32 pair-units), one pair-unit per lane, so a wide
// row (a query row of 32 heads) spreads over several warps.
template <int STYLE>
__global__ void __launch_bounds__(256) rope_rows_kernel(uint8_t* out, const uint8_t* x, RowMap imap,
                                                        RowMap omap, const int32_t* pos_from,
                                                        const int32_t* pos_to, int32_t* pos_out, int n,
                                                        int n_heads, int head_dim, RopeTable t,
                                                        int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const int units = n_heads * head_dim / (STYLE == 0 ? 16 : 8);
  const int per_row = (units + kWarp - 1) / kWarp;
  const long long items = (long long)n * per_row;
  const long long warps = (long long)gridDim.x * (blockDim.x / kWarp);
  const size_t row_bytes = (size_t)n_heads * head_dim * 2;
  const int half = head_dim / 2;
  for (long long item = blockIdx.x * (long long)(blockDim.x / kWarp) + threadIdx.x / kWarp; item < items;
       item += warps) {
    const int i = (int)(item / per_row);
    const int u = (int)(item % per_row) * kWarp + lane;
    const int src_row = map_row(imap, i);
    const int dst_row = map_row(omap, i);
    const int to = pos_to ? pos_to[i] : src_row;
    const int from = pos_from ? pos_from[i] : 0;
    const int delta = to - from;
    const int ad = delta < 0 ? -delta : delta;
    const bool first = item % per_row == 0 && lane == 0;
    if (pos_out && first) pos_out[i] = to;
    if (src_row < 0 || dst_row < 0 || src_row >= imap.limit || dst_row >= omap.limit) {
      if (first) record_error(err, kErrIndex, i);
      continue;
    }
    if (ad >= t.len) {
      if (first) record_error(err, kErrRopeRange, i);
      continue;
    }
    if (u < units)
      rotate_unit<STYLE>(out + dst_row * row_bytes, x + src_row * row_bytes, u, head_dim,
                         t.tab + (size_t)ad * half, delta < 0);
  }
}

// ---------------------------------------------------------------------------
// Deviation, canonical order: lane l sums chunks l, l+32, ... (8 elements each) as
// acc = fl(acc + fl(d*d)), then a xor butterfly over the lanes.
//   V only (KS < 0):  d = fl(v_new - v_old).
//   K+V (KS = RoPE style): first the key part, d = fl(x' - k_old) where x' is the recomputed
//   key turned to the token's chunk-local position p_old = t mod chunk_len in fp32 from the
//   table row of p_old (first pair member x' = fl(fl(x c) - fl(y s)), second member
//   y' = fl(fl(x s) + fl(y c))); then the V part. Each lane adds all its key chunks before
//   its V chunks. Products and sums are separately rounded (no fused multiply-add).
// Candidate i's deviation (one warp): the body of kv_deviation_kernel and of its batched form.
template <int CPL, int KS>
__device__ __forceinline__ void deviation_row(const uint8_t* k_new, const uint8_t* k_old, const uint8_t* v_new,
                                              const uint8_t* v_old, const int32_t* cand, int i, int n_rows,
                                              int elems, int head_dim, int chunk_len, RopeTable tab, float* dev,
                                              int32_t* err) {
  const int lane = threadIdx.x % kWarp;
  const int t = cand ? cand[i] : i;
  if (t < 0 || t >= n_rows) {
    if (lane == 0) {
      dev[i] = __int_as_float(0x7fc00000);
      record_error(err, kErrIndex, i);
    }
    return;
  }
  const int chunks = elems / 8;
  const size_t row_bytes = (size_t)elems * 2;
  float acc = 0.0f;
  if constexpr (KS >= 0) {
    const uint8_t* kn = k_new + (size_t)t * row_bytes;
    const uint8_t* ko = k_old + (size_t)t * row_bytes;
    const float2* cs = tab.tab + (size_t)(t % chunk_len) * (head_dim / 2);
    const int per_head = head_dim / 8;  // chunks per head
    uint4 a[CPL], b[CPL], pa[CPL];
#pragma unroll
    for (int r = 0; r < CPL; ++r) {
      const int c = lane + kWarp * r;
      if (c < chunks) {
        a[r] = ld_stream(kn + (size_t)c * 16);
        b[r] = ld_stream(ko + (size_t)c * 16);
        if (KS == 0) {  // the other members of the chunk's pairs sit D/2 elements away
          const int ch = c % per_head;
          pa[r] = ld_stream(kn + (size_t)(ch < per_head / 2 ? c + per_head / 2 : c - per_head / 2) * 16);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < CPL; ++r) {
      const int c = lane + kWarp * r;
      if (c < chunks) {
        float x[8], o[8];
        unpack8(a[r], x);
        unpack8(b[r], o);
        const int ch = c % per_head;
        if (KS == 0) {
          float y[8];
          unpack8(pa[r], y);
          const bool first = ch < per_head / 2;
          const float4* t4 = reinterpret_cast<const float4*>(cs + (first ? ch : ch - per_head / 2) * 8);
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const float4 q = __ldg(t4 + e2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * e2 + h;
              const float c0 = h ? q.z : q.x, s0 = h ? q.w : q.y;
              const float rot = first ? __fsub_rn(__fmul_rn(x[e], c0), __fmul_rn(y[e], s0))
                                      : __fadd_rn(__fmul_rn(y[e], s0), __fmul_rn(x[e], c0));
              const float d = __fsub_rn(rot, o[e]);
              acc = __fadd_rn(acc, __fmul_rn(d, d));
            }
          }
        } else {
          const float4* t4 = reinterpret_cast<const float4*>(cs + ch * 4);
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const float4 q = __ldg(t4 + e2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 4 * e2 + 2 * h;
              const float c0 = h ? q.z : q.x, s0 = h ? q.w : q.y;
              const float r0 = __fsub_rn(__fmul_rn(x[e], c0), __fmul_rn(x[e + 1], s0));
              const float r1 = __fadd_rn(__fmul_rn(x[e], s0), __fmul_rn(x[e + 1], c0));
              const float d0 = __fsub_rn(r0, o[e]);
              acc = __fadd_rn(acc, __fmul_rn(d0, d0));
              const float d1 = __fsub_rn(r1, o[e + 1]);
              acc = __fadd_rn(acc, __fmul_rn(d1, d1));
            }
          }
        }
      }
    }
  }
  const uint8_t* pn = v_new + (size_t)t * row_bytes;
  const uint8_t* po = v_old + (size_t)t * row_bytes;
  uint4 a[CPL], b[CPL];
#pragma unroll
  for (int r = 0; r < CPL; ++r) {
    const int c = lane + kWarp * r;
    if (c < chunks) {
      a[r] = ld_stream(pn + (size_t)c * 16);
      b[r] = ld_stream(po + (size_t)c * 16);
    }
  }
#pragma unroll
  for (int r = 0; r < CPL; ++r) {
    const int c = lane + kWarp * r;
    if (c < chunks) {
      float x[8], y[8];
      unpack8(a[r], x);
      unpack8(b[r], y);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = __fsub_rn(x[e], y[e]);
        acc = __fadd_rn(acc, __fmul_rn(d, d));
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
  if (lane == 0) dev[i] = acc;
}

template <int CPL, int KS>
__global__ void __launch_bounds__(256) kv_deviation_kernel(const uint8_t* k_new, const uint8_t* k_old,
                                                           const uint8_t* v_new, const uint8_t* v_old,
                                                           const int32_t* cand, int m, int n_rows, int elems,
                                                           int head_dim, int chunk_len, RopeTable tab, float* dev,
                                                           int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  if (i >= m) return;
  deviation_row<CPL, KS>(k_new, k_old, v_new, v_old, cand, i, n_rows, elems, head_dim, chunk_len, tab, dev, err);
}

// The deviations of several layers over one candidate list (blockIdx.y = layer of the batch).
template <int CPL, int KS>
__global__ void __launch_bounds__(256) kv_deviation_batch_kernel(const __grid_constant__ SelectBatch b,
                                                                 const int32_t* cand, int m, int n_rows, int elems,
                                                                 int head_dim, int chunk_len, RopeTable tab,
                                                                 int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  const int l = blockIdx.y;
  if (i >= m || l >= b.n) return;
  deviation_row<CPL, KS>((const uint8_t*)b.k_new[l], (const uint8_t*)b.k_old[l], (const uint8_t*)b.v_new[l],
                         (const uint8_t*)b.v_old[l], cand, i, n_rows, elems, head_dim, chunk_len, tab, b.dev[l], err);
}

// ---------------------------------------------------------------------------
// Top-k by MSB-first 8-bit radix select on order-preserving keys, then a
// stable compaction. One block of 1024 threads.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkThreads = 1024;

// The selection of one list by one block of kTopkThreads: the body of hkvd_topk_kernel and of its
// batched form.
__device__ __forceinline__ void topk_block(const float* __restrict__ dev, const int32_t* __restrict__ cand, int m,
                                           int k, int32_t* sel_tok, int32_t* sel_row, int32_t* err) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_remaining;
  __shared__ int warp_eq[32], warp_sel[32], warp_eq_ex[32], warp_sel_ex[32];
  __shared__ int s_base_eq, s_base_sel, s_tile_eq, s_tile_sel;
  const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
  if (tid == 0) {
    s_prefix = 0;
    s_mask = 0;
    s_remaining = k;
    s_base_eq = 0;
    s_base_sel = 0;
  }
  // candidate ids must be strictly ascending (the output order relies on it)
  if (cand) {
    for (int i = tid; i + 1 < m; i += kTopkThreads)
      if (cand[i] >= cand[i + 1]) record_error(err, kErrOrder, i);
  }
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int d = tid; d < 256; d += kTopkThreads) hist[d] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int i = tid; i < m; i += kTopkThreads) {
      const uint32_t key = order_key(dev[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits [248 - 8l, 256 - 8l), scanned from the top digit down
      uint32_t c[8];
      uint32_t sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = hist[255 - 8 * lane - e];
        sum += c[e];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const uint32_t before = incl - sum;
      const uint32_t need = (uint32_t)s_remaining;
      if (before < need && need <= incl) {
        uint32_t cum = before;
        for (int e = 0; e < 8; ++e) {
          if (cum + c[e] >= need) {
            const uint32_t digit = 255u - 8u * lane - e;
            s_prefix = prefix | (digit << shift);
            s_mask = mask | (255u << shift);
            s_remaining = (int)(need - cum);
            break;
          }
          cum += c[e];
        }
      }
    }
    __syncthreads();
  }
  const uint32_t thr = s_prefix;
  const int need_eq = s_remaining;  // keys equal to thr to keep, lowest rows first
  const uint32_t below = (1u << lane) - 1u;
  for (int base = 0; base < m; base += kTopkThreads) {
    const int i = base + tid;
    const uint32_t key = i < m ? order_key(dev[i]) : 0u;
    const bool gt = i < m && key > thr;
    const bool eq = i < m && key == thr;
    const uint32_t eq_mask = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_eq[warp] = __popc(eq_mask);
    __syncthreads();
    if (warp == 0) {
      const int v = warp_eq[lane];
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
      }
      warp_eq_ex[lane] = incl - v;
      if (lane == 31) s_tile_eq = incl;
    }
    __syncthreads();
    const int eq_rank = s_base_eq + warp_eq_ex[warp] + __popc(eq_mask & below);
    const bool sel = gt || (eq && eq_rank < need_eq);
    const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) warp_sel[warp] = __popc(sel_mask);
    __syncthreads();
    if (warp == 0) {
      const int v = warp_sel[lane];
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
      }
      warp_sel_ex[lane] = incl - v;
      if (lane == 31) s_tile_sel = incl;
    }
    __syncthreads();
    if (sel) {
      const int pos = s_base_sel + warp_sel_ex[warp] + __popc(sel_mask & below);
      if (pos < k) {
        sel_tok[pos] = cand ? cand[i] : i;
        sel_row[pos] = i;
      }
    }
    __syncthreads();
    if (tid == 0) {
      s_base_eq += s_tile_eq;
      s_base_sel += s_tile_sel;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kTopkThreads) hkvd_topk_kernel(const float* __restrict__ dev,
                                                                  const int32_t* __restrict__ cand, int m,
                                                                  int k, int32_t* sel_tok, int32_t* sel_row,
                                                                  int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  topk_block(dev, cand, m, k, sel_tok, sel_row, err);
}

// The selections of several layers over one candidate list (block l = layer l of the batch).
__global__ void __launch_bounds__(kTopkThreads) hkvd_topk_batch_kernel(const __grid_constant__ SelectBatch b,
                                                                        const int32_t* __restrict__ cand, int m,
                                                                        int k, int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int l = blockIdx.x;
  if (l >= b.n) return;
  topk_block(b.dev[l], cand, m, k, b.sel_tok[l], b.sel_row[l], err);
}

// ---------------------------------------------------------------------------
// Fused cache: kFuseRows consecutive rows per block, one warp per row, at most 64 registers a
// thread. On the large layers whose attention runs the paired-tile kernel the pass uses 2-row
// blocks: four times the blocks stream the layer faster (the long-context request's fuse in 55.4
// against 57.7 us, 0.958 against 0.921 of the copy bandwidth), and none of them can sit beside a
// paired-tile CTA, which holds all of an SM's registers. Beside the one-tile kernel, which leaves
// room for fuse blocks, the 8-row blocks stay: 2-row blocks there slowed the Mistral-7B step by 9%.
constexpr int kFuseRowsWide = 8;
constexpr int kFuseRowsNarrow = 2;
constexpr int kFuseThreads = 256;  // the standalone scatter
constexpr int kQParts = 4;  // warps per query row in the fused pass

// First index j in the ascending list sel[0..k) with sel[j] >= key (k if none),
// by one warp: 32-ary search, one coalesced probe and ballot per round.
__device__ __forceinline__ int warp_lower_bound(const int32_t* sel, int k, int key, int lane) {
  int lo = 0, hi = k;  // the answer lies in [lo, hi]
  while (hi - lo > kWarp) {
    const int step = (hi - lo + kWarp - 1) / kWarp;
    const int idx = lo + lane * step;
    const unsigned less = __ballot_sync(0xffffffffu, idx < hi && sel[idx] < key);
    const int c = __popc(less);  // probes below the answer form a prefix of the lanes
    if (c == 0) {
      hi = lo;
      break;
    }
    const int nlo = lo + (c - 1) * step + 1;
    hi = min(hi, lo + c * step);
    lo = nlo;
  }
  const int idx = lo + lane;
  return lo + __popc(__ballot_sync(0xffffffffu, idx < hi && sel[idx] < key));
}

// Blocks [0, ceil(n_tokens / 8)) build the fused K/V rows; the blocks after them
// encode the query rows (one warp per row), so the layer's streaming work is
// one launch.
template <int STYLE, int kFuseRows>
__global__ void __maxnreg__(64) blend_fuse_kernel(
    uint8_t* k_fused, uint8_t* v_fused, const uint8_t* k_old, const uint8_t* v_old, const uint8_t* k_new,
    const uint8_t* v_new, const int32_t* sel, int k, int32_t* out_tok, int32_t* out_row, int n_ctx,
    int chunk_len, int n_tokens, int hkv, int head_dim, RopeTable t, const uint8_t* q, uint8_t* q_rot, int mq,
    int hq, int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint8_t is_sel[kFuseRows];
  const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
  const int kv_blocks = (n_tokens + kFuseRows - 1) / kFuseRows;
  if ((int)blockIdx.x >= kv_blocks) {
    // query row i: token sel[i] (i < k) or n_ctx + i - k, encoded at its own position; a row is
    // shared by kQParts warps (each a contiguous group of heads), so every warp has one batch of
    // loads in flight instead of several in turn
    const int qw = ((int)blockIdx.x - kv_blocks) * kFuseRows + warp;
    const int parts = (hq % kQParts == 0) ? kQParts : 1;
    const int i = qw / kQParts, part = qw % kQParts;
    if (i >= mq || part >= parts) return;
    const int tok = i < k ? sel[i] : n_ctx + (i - k);
    if (tok < 0 || tok >= n_tokens || (i < k && tok >= n_ctx)) {
      if (lane == 0) record_error(err, kErrIndex, i);
      return;
    }
    if (tok >= t.len) {
      if (lane == 0) record_error(err, kErrRopeRange, tok);
      return;
    }
    const size_t q_bytes = (size_t)hq * head_dim * 2;
    const int part_heads = hq / parts;
    const size_t part_off = (size_t)part * part_heads * head_dim * 2;
    rotate_row<STYLE, 2>(q_rot + (size_t)i * q_bytes + part_off, q + (size_t)tok * q_bytes + part_off, part_heads,
                         head_dim, t.tab + (size_t)tok * (head_dim / 2), false, lane);
    return;
  }
  // A suffix row's source does not depend on the selection (always recomputed): pull its lines
  // into L2 while warp 0 reads the list. A context row's source is known only after the list
  // is read (prefetching the cached row would read a selected row's lines for nothing).
  {
    const int tok = blockIdx.x * kFuseRows + warp;
    if (tok >= n_ctx && tok < n_tokens) {
      const size_t rb = (size_t)hkv * head_dim * 2;
      const uint8_t* kp = k_new + tok * rb;
      const uint8_t* vp = v_new + tok * rb;
      for (size_t off = (size_t)lane * 128; off < rb; off += 32 * 128) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(kp + off));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(vp + off));
      }
    }
  }
  const int r0 = blockIdx.x * kFuseRows;
  if (out_tok != nullptr && threadIdx.x < kFuseRows) {
    // a layer that keeps its candidates: S = C is copied out alongside the pass
    const int i = r0 + threadIdx.x;
    if (i < k) {
      out_tok[i] = sel[i];
      out_row[i] = i;
    }
  }
  if (warp == 0) {
    const int j0 = warp_lower_bound(sel, k, r0, lane);
    if (lane < kFuseRows) {
      is_sel[lane] = 0;
      __syncwarp((1u << kFuseRows) - 1);
      const int j = j0 + lane;
      if (j < k) {
        const int tk = sel[j];
        if (tk < 0 || tk >= n_ctx) record_error(err, kErrIndex, j);
        else if (j > 0 && sel[j - 1] >= tk) record_error(err, kErrOrder, j);
        else if (tk < r0 + kFuseRows) is_sel[tk - r0] = 1;
      }
    }
  }
  __syncthreads();
  const int tok = r0 + warp;
  if (tok >= n_tokens) return;
  const size_t row_bytes = (size_t)hkv * head_dim * 2;
  const bool fresh = tok >= n_ctx || is_sel[warp];
  const int pos = fresh ? tok : (tok / chunk_len) * chunk_len;  // encode at p, or move by the chunk start
  if (pos >= t.len) {
    if (lane == 0) record_error(err, kErrRopeRange, tok);
    return;
  }
  const uint8_t* ks = (fresh ? k_new : k_old) + tok * row_bytes;
  const uint8_t* vs = (fresh ? v_new : v_old) + tok * row_bytes;
  rotate_row<STYLE, 2>(k_fused + tok * row_bytes, ks, hkv, head_dim, t.tab + (size_t)pos * (head_dim / 2), false,
                       lane);
  copy_row(v_fused + tok * row_bytes, vs, (int)row_bytes, lane);
}

template <int STYLE>
__global__ void __launch_bounds__(kFuseThreads) fuse_scatter_kernel(uint8_t* k_fused, uint8_t* v_fused,
                                                                    const uint8_t* k_new, const uint8_t* v_new,
                                                                    const int32_t* sel, int k, int n_ctx,
                                                                    int n_tokens, int hkv, int head_dim,
                                                                    RopeTable t, int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const int warps = gridDim.x * (blockDim.x / kWarp);
  const int rows = k + (n_tokens - n_ctx);
  const size_t row_bytes = (size_t)hkv * head_dim * 2;
  const int half = head_dim / 2;
  for (int i = blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; i < rows; i += warps) {
    const int tok = i < k ? sel[i] : n_ctx + (i - k);
    if (tok < 0 || tok >= n_tokens || (i < k && tok >= n_ctx) || (i > 0 && i < k && sel[i - 1] >= tok)) {
      if (lane == 0) record_error(err, i < k && i > 0 && tok < n_ctx && tok >= 0 ? kErrOrder : kErrIndex, i);
      continue;
    }
    if (tok >= t.len) {
      if (lane == 0) record_error(err, kErrRopeRange, tok);
      continue;
    }
    rotate_row<STYLE, 2>(k_fused + tok * row_bytes, k_new + tok * row_bytes, hkv, head_dim,
                         t.tab + (size_t)tok * half, false, lane);
    copy_row(v_fused + tok * row_bytes, v_new + tok * row_bytes, (int)row_bytes, lane);
  }
}

int grid_for_warps(long long warps_needed, int warps_per_block) {
  long long b = (warps_needed + warps_per_block - 1) / warps_per_block;
  if (b < 1) b = 1;
  if (b > 152LL * 64) b = 152LL * 64;
  return (int)b;
}

}  // namespace

cudaError_t launch_rope_rows(void* out, const void* x, RowMap imap, RowMap omap, const int32_t* pos_from,
                             const int32_t* pos_to, int32_t* pos_out, int32_t n, int32_t n_heads,
                             int32_t head_dim, int32_t style, RopeTable t, int32_t* err, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int units = n_heads * head_dim / (style == 0 ? 16 : 8);
  const int grid = grid_for_warps((long long)n * ((units + kWarp - 1) / kWarp), 8);
  if (style == 0)
    return launch_pdl(rope_rows_kernel<0>, grid, 256, 0, s, (uint8_t*)out, (const uint8_t*)x, imap, omap,
                      pos_from, pos_to, pos_out, n, n_heads, head_dim, t, err);
  else
    return launch_pdl(rope_rows_kernel<1>, grid, 256, 0, s, (uint8_t*)out, (const uint8_t*)x, imap, omap,
                      pos_from, pos_to, pos_out, n, n_heads, head_dim, t, err);
  return cudaPeekAtLastError();
}

template <int KS>
static cudaError_t launch_kv_deviation_t(const void* k_new, const void* k_old, const void* v_new, const void* v_old,
                                        const int32_t* cand, int32_t m, int32_t n_rows, int32_t hkv,
                                        int32_t head_dim, int32_t chunk_len, RopeTable t, float* dev, int32_t* err,
                                        cudaStream_t s) {
  const int elems = hkv * head_dim;
  const int cpl = (elems + 255) / 256;
  const int grid = (m + 7) / 8;
  const auto* kn = (const uint8_t*)k_new;
  const auto* ko = (const uint8_t*)k_old;
  const auto* vn = (const uint8_t*)v_new;
  const auto* vo = (const uint8_t*)v_old;
#define CB_DEV_LAUNCH(C)                                                                                      \
  return launch_pdl(kv_deviation_kernel<C, KS>, grid, 256, 0, s, kn, ko, vn, vo, cand, m, n_rows, elems, head_dim, \
                    chunk_len, t, dev, err)
  if (cpl <= 1) CB_DEV_LAUNCH(1);
  if (cpl <= 2) CB_DEV_LAUNCH(2);
  if (cpl <= 4) CB_DEV_LAUNCH(4);
  if (cpl <= 8) CB_DEV_LAUNCH(8);
#undef CB_DEV_LAUNCH
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_deviation(const void* k_new, const void* k_old, const void* v_new, const void* v_old,
                                const int32_t* cand, int32_t m, int32_t n_rows, int32_t hkv, int32_t head_dim,
                                int32_t chunk_len, int32_t style, RopeTable t, float* dev, int32_t* err,
                                cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  if (k_new == nullptr)
    return launch_kv_deviation_t<-1>(nullptr, nullptr, v_new, v_old, cand, m, n_rows, hkv, head_dim, 1, t, dev, err,
                                     s);
  if (style == 0)
    return launch_kv_deviation_t<0>(k_new, k_old, v_new, v_old, cand, m, n_rows, hkv, head_dim, chunk_len, t, dev,
                                    err, s);
  return launch_kv_deviation_t<1>(k_new, k_old, v_new, v_old, cand, m, n_rows, hkv, head_dim, chunk_len, t, dev, err,
                                  s);
}

template <int KS>
static cudaError_t launch_select_batch_t(const SelectBatch& b, const int32_t* cand, int32_t m, int32_t k,
                                         int32_t n_rows, int32_t hkv, int32_t head_dim, int32_t chunk_len,
                                         RopeTable t, int32_t* err, cudaStream_t s) {
  const int elems = hkv * head_dim;
  const int cpl = (elems + 255) / 256;
  const dim3 grid((m + 7) / 8, b.n);
  cudaError_t e;
#define CB_DEVB_LAUNCH(C) \
  e = launch_pdl(kv_deviation_batch_kernel<C, KS>, grid, 256, 0, s, b, cand, m, n_rows, elems, head_dim, chunk_len, t, err)
  if (cpl <= 1)
    CB_DEVB_LAUNCH(1);
  else if (cpl <= 2)
    CB_DEVB_LAUNCH(2);
  else if (cpl <= 4)
    CB_DEVB_LAUNCH(4);
  else
    CB_DEVB_LAUNCH(8);
#undef CB_DEVB_LAUNCH
  if (e != cudaSuccess || k <= 0) return e;
  return launch_pdl(hkvd_topk_batch_kernel, b.n, kTopkThreads, 0, s, b, cand, m, k, err);
}

cudaError_t launch_select_batch(const SelectBatch& b, const int32_t* cand, int32_t m, int32_t k, int32_t n_rows,
                                int32_t hkv, int32_t head_dim, int32_t chunk_len, int32_t style, RopeTable t,
                                int32_t* err, cudaStream_t s) {
  if (m <= 0 || b.n <= 0) return cudaSuccess;
  if (b.n > kSelectBatchMax) return cudaErrorInvalidValue;
  if (b.k_new[0] == nullptr) return launch_select_batch_t<-1>(b, cand, m, k, n_rows, hkv, head_dim, 1, t, err, s);
  if (style == 0) return launch_select_batch_t<0>(b, cand, m, k, n_rows, hkv, head_dim, chunk_len, t, err, s);
  return launch_select_batch_t<1>(b, cand, m, k, n_rows, hkv, head_dim, chunk_len, t, err, s);
}

cudaError_t launch_hkvd_topk(const float* dev, const int32_t* cand, int32_t m, int32_t k, int32_t* sel_tok,
                             int32_t* sel_row, int32_t* err, cudaStream_t s) {
  if (k <= 0 || m <= 0) return cudaSuccess;
  return launch_pdl(hkvd_topk_kernel, 1, kTopkThreads, 0, s, dev, cand, m, k, sel_tok, sel_row, err);
}

cudaError_t launch_fuse_scatter(void* k_fused, void* v_fused, const void* k_new, const void* v_new,
                                const int32_t* sel_tok, int32_t k, int32_t n_ctx, int32_t n_tokens,
                                int32_t hkv, int32_t head_dim, int32_t style, RopeTable t, int32_t* err,
                                cudaStream_t s) {
  const int rows = k + (n_tokens - n_ctx);
  if (rows <= 0) return cudaSuccess;
  const int grid = grid_for_warps(rows, kFuseThreads / kWarp);
  if (style == 0)
    return launch_pdl(fuse_scatter_kernel<0>, grid, kFuseThreads, 0, s, (uint8_t*)k_fused, (uint8_t*)v_fused,
                      (const uint8_t*)k_new, (const uint8_t*)v_new, sel_tok, k, n_ctx, n_tokens, hkv, head_dim, t,
                      err);
  else
    return launch_pdl(fuse_scatter_kernel<1>, grid, kFuseThreads, 0, s, (uint8_t*)k_fused, (uint8_t*)v_fused,
                      (const uint8_t*)k_new, (const uint8_t*)v_new, sel_tok, k, n_ctx, n_tokens, hkv, head_dim, t,
                      err);
  return cudaPeekAtLastError();
}

cudaError_t launch_blend_fuse(void* k_fused, void* v_fused, const void* k_old, const void* v_old,
                              const void* k_new, const void* v_new, const int32_t* sel_tok, int32_t k,
                              int32_t* copy_tok, int32_t* copy_row, int32_t n_ctx, int32_t chunk_len,
                              int32_t n_tokens, int32_t hkv, int32_t head_dim, int32_t style, RopeTable t,
                              const void* q, void* q_rot, int32_t mq, int32_t hq, bool narrow, int32_t* err,
                              cudaStream_t s) {
  if (n_tokens <= 0) return cudaSuccess;
  if (q == nullptr || q_rot == nullptr) mq = 0;
  const int rows = narrow ? kFuseRowsNarrow : kFuseRowsWide;
  const int grid = (n_tokens + rows - 1) / rows + (mq * kQParts + rows - 1) / rows;
  auto* kf = (uint8_t*)k_fused;
  auto* vf = (uint8_t*)v_fused;
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, grid, rows * kWarp, 0, s, kf, vf, (const uint8_t*)k_old, (const uint8_t*)v_old,
                      (const uint8_t*)k_new, (const uint8_t*)v_new, sel_tok, k, copy_tok, copy_row, n_ctx, chunk_len,
                      n_tokens, hkv, head_dim, t, (const uint8_t*)q, (uint8_t*)q_rot, mq, hq, err);
  };
  if (style == 0)
    return narrow ? go(blend_fuse_kernel<0, kFuseRowsNarrow>) : go(blend_fuse_kernel<0, kFuseRowsWide>);
  return narrow ? go(blend_fuse_kernel<1, kFuseRowsNarrow>) : go(blend_fuse_kernel<1, kFuseRowsWide>);
}


}  // namespace cb
