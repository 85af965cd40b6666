// Decode attention over a (blended) KV cache: the newest token is the only query row
// ("rag的kvcache问题" §阶段 2 (Decode): a [1, d] query against the whole cache, memory-bound).
//
// out[h] = sum_{j < n_keys} softmax_j(scale q[h] . k[j, g]) v[j, g],  g = h / G.
//
// HBM-bound: every key costs 2 * D * 2 bytes per kv head and 4 * G * D flops, so the
// kernel streams K and V once on the CUDA cores (tensor cores would idle on a G-row
// problem). Grid (splits, Hkv), about two CTAs of 8 warps per SM: a CTA takes a contiguous
// key range of one kv head; its warps take groups of KEYS keys in turn, lane l holding
// dims [l * D/32, (l + 1) * D/32) of each key, with the next group's rows in flight while
// the current one is computed. Per group a lane forms its partial dot products for every
// (key, head) pair and a recursive-halving shuffle reduction leaves lane l the whole score
// of one pair; the per-head max runs over the lanes of that head, each lane exponentiates
// its own score, and the weights pass through a per-warp shared array to every lane, which
// updates its slice of the G output rows (online softmax in the log2 domain). The warps
// merge in a fixed order in shared memory; each CTA writes (max, sum, unnormalised rows)
// to the plan's scratch, and the last CTA of the kv head to finish (a ticket counter)
// merges the splits, with all its loads issued before the arithmetic.
#include "common.cuh"
#include "kernels.h"

namespace cb {

namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;

// Keys per warp step: 8 keys, fewer for large groups so that a lane keeps at most 32 partial sums.
template <int G>
__host__ __device__ constexpr int dec_keys() {
  return G >= 16 ? 2 : (G >= 8 ? 4 : 8);
}

template <int DPL>
struct KvLane;  // one lane's slice (DPL bf16) of one key or value row
template <>
struct KvLane<4> {
  uint2 v;
  __device__ __forceinline__ void load(const uint8_t* p) {
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  }
  __device__ __forceinline__ void zero() { v = make_uint2(0u, 0u); }
  __device__ __forceinline__ void unpack(float f[4]) const {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
};
template <>
struct KvLane<2> {
  uint32_t v;
  __device__ __forceinline__ void load(const uint8_t* p) {
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  }
  __device__ __forceinline__ void zero() { v = 0u; }
  __device__ __forceinline__ void unpack(float f[2]) const {
    f[0] = __uint_as_float(v << 16); f[1] = __uint_as_float(v & 0xffff0000u);
  }
};

constexpr int kDecMaxSplits = 40;  // splits per kv head

// L2 loads of other CTAs' partials (not cached in L1; ordered after the ticket by the fence).
__device__ __forceinline__ float2 ld_cg(const float2* p) {
  float2 v;
  asm("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ld_cg(const float4* p) {
  float4 v;
  asm("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 2) decode_attention_kernel(const uint8_t* __restrict__ q,
                                                                       const uint8_t* __restrict__ k,
                                                                       const uint8_t* __restrict__ v, int n_keys,
                                                                       int hkv, int per_split, float qscale,
                                                                       float* part_o, float2* part_ml,
                                                                       int32_t* tickets, uint8_t* out) {
  constexpr int DPL = D / 32;
  constexpr int KEYS = dec_keys<G>();
  constexpr int NV = KEYS * G;               // (key, head) pairs per step
  constexpr int SHIFT = NV >= 32 ? 0 : (NV == 16 ? 1 : (NV == 8 ? 2 : 3));
  static_assert(NV == 8 || NV == 16 || NV == 32, "unsupported group size");
  // lane bits: [0, SHIFT) replicate one pair, [SHIFT, SHIFT + LG) its head, the rest its key
  constexpr int LG = G == 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : (G == 8 ? 3 : 4)));
  constexpr int KEY_BIT0 = SHIFT + LG;

  __shared__ __align__(16) float s_p[kDecWarps][NV];  // a step's weights, read by every lane
  __shared__ __align__(16) float s_a[kDecWarps][G > 4 ? G : 4];  // a step's rescale factor per head
  __shared__ float s_m[kDecWarps][G], s_l[kDecWarps][G];
  __shared__ float s_o[kDecWarps / 2][G][D];
  __shared__ float s_w[kDecMaxSplits][G];  // merge: weight of split s for head h
  __shared__ int s_last;

  pdl_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = blockIdx.y, split = blockIdx.x, n_split = gridDim.x;
  const int k0 = split * per_split;
  const int k1 = min(n_keys, k0 + per_split);
  const int my_pair = lane >> SHIFT;  // (key, head) pair whose score this lane holds
  const int my_head = my_pair % G, my_key = my_pair / G;
  const size_t row = (size_t)hkv * D * 2;  // bytes per key row
  const uint8_t* kb = k + (size_t)g * D * 2 + lane * DPL * 2;
  const uint8_t* vb = v + (size_t)g * D * 2 + lane * DPL * 2;
  pdl_wait();

  float m_my = -INFINITY, l_my = 0.0f;  // running max and sum of this lane's head (its keys)
  float o[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.0f;

  const int stride = kDecWarps * KEYS;
  KvLane<DPL> kc[KEYS], vc[KEYS], kn[KEYS], vn[KEYS];
  auto load_step = [&](KvLane<DPL>* kk, KvLane<DPL>* vv, int j) {
#pragma unroll
    for (int i = 0; i < KEYS; ++i) {
      if (j + i < k1) {
        kk[i].load(kb + (size_t)(j + i) * row);
        vv[i].load(vb + (size_t)(j + i) * row);
      } else {
        kk[i].zero();
        vv[i].zero();
      }
    }
  };
  int j = k0 + warp * KEYS;
  if (j < k1) load_step(kc, vc, j);  // the first rows are requested before the query

  // this lane's query slice of the G heads, scaled into the log2 domain
  float qf[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    KvLane<DPL> t;
    t.load(q + ((size_t)(g * G + h) * D + lane * DPL) * 2);
    t.unpack(qf[h]);
#pragma unroll
    for (int e = 0; e < DPL; ++e) qf[h][e] *= qscale;
  }

  for (; j < k1; j += stride) {
    if (j + stride < k1) load_step(kn, vn, j + stride);  // next step's rows in flight during this one

    // partial dot products of this lane's dims: x[i * G + h]
    float x[NV];
#pragma unroll
    for (int i = 0; i < KEYS; ++i) {
      float kf[DPL];
      kc[i].unpack(kf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float acc = qf[h][0] * kf[0];
#pragma unroll
        for (int e = 1; e < DPL; ++e) acc = fmaf(qf[h][e], kf[e], acc);
        x[i * G + h] = acc;
      }
    }
    // recursive halving over the lanes: after offset o the lane keeps the half of its values
    // selected by its lane bit o, so lane l ends with the whole score of pair l >> SHIFT
    // (fewer than 32 pairs: the last offsets sum replicated copies).
    int cnt = NV;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      if (cnt > 1) {
        const int half = cnt / 2;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int t = 0; t < NV / 2; ++t) {
          if (t < half) {
            const float send = upper ? x[t] : x[t + half];
            const float keep = upper ? x[t + half] : x[t];
            x[t] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
        }
        cnt = half;
      } else {
        x[0] += __shfl_xor_sync(0xffffffffu, x[0], off);
      }
    }
    // online softmax: the max over the lanes of this head, one exponential per lane
    const float sc = (j + my_key < k1) ? x[0] : -INFINITY;
    float mx = sc;
#pragma unroll
    for (int off = 1 << KEY_BIT0; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m_my, mx);  // finite: a step holds at least one key in range
    const float alpha = exp2f(m_my - m_new);
    const float p = exp2f(sc - m_new);
    m_my = m_new;
    l_my = fmaf(l_my, alpha, p);
    if ((lane & ((1 << SHIFT) - 1)) == 0) s_p[warp][my_pair] = p;
    if (my_key == 0 && (lane & ((1 << SHIFT) - 1)) == 0) s_a[warp][my_head] = alpha;
    __syncwarp();
    // this lane's slice of the output rows
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float a = s_a[warp][h];
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[h][e] *= a;
    }
#pragma unroll
    for (int i = 0; i < KEYS; ++i) {
      float vf[DPL];
      vc[i].unpack(vf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pw = s_p[warp][i * G + h];
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pw, vf[e], o[h][e]);
      }
    }
    __syncwarp();  // the next step rewrites s_p / s_a
#pragma unroll
    for (int i = 0; i < KEYS; ++i) {
      kc[i] = kn[i];
      vc[i] = vn[i];
    }
  }

  // per-warp max and sum of each head: the lanes of head h hold them for its keys
#pragma unroll
  for (int off = 1 << KEY_BIT0; off < 32; off <<= 1) l_my += __shfl_xor_sync(0xffffffffu, l_my, off);
  if (my_key == 0 && (lane & ((1 << SHIFT) - 1)) == 0) {
    s_m[warp][my_head] = m_my;
    s_l[warp][my_head] = l_my;
  }
  __syncthreads();
  // merge the warps in a fixed order (a warp or CTA without keys has max -inf and sum 0):
  // rescale every warp to the CTA's max, warps 4-7 add onto warps 0-3, then sum 0-3.
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mm = s_m[0][h];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) mm = fmaxf(mm, s_m[w][h]);
    const float a = s_m[warp][h] == -INFINITY ? 0.0f : exp2f(s_m[warp][h] - mm);
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] *= a;
  }
  constexpr int kHalf = kDecWarps / 2;
  if (warp < kHalf) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) s_o[warp][h][lane * DPL + e] = o[h][e];
  }
  __syncthreads();
  if (warp >= kHalf) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) s_o[warp - kHalf][h][lane * DPL + e] += o[h][e];
  }
  __syncthreads();
  constexpr int kOut = G * D;
  for (int idx = threadIdx.x; idx < kOut; idx += kDecThreads) {
    const int h = idx / D, d = idx % D;
    float oo = s_o[0][h][d];
#pragma unroll
    for (int w = 1; w < kHalf; ++w) oo += s_o[w][h][d];
    float mm = s_m[0][h];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) mm = fmaxf(mm, s_m[w][h]);
    float ll = 0.0f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) ll = fmaf(s_m[w][h] == -INFINITY ? 0.0f : exp2f(s_m[w][h] - mm), s_l[w][h], ll);
    if (n_split == 1) {
      reinterpret_cast<__nv_bfloat16*>(out)[(size_t)(g * G + h) * D + d] = __float2bfloat16_rn(oo / ll);
    } else {
      const size_t unit = (size_t)g * n_split + split;
      part_o[(unit * G + h) * D + d] = oo;
      if (d == 0) part_ml[unit * G + h] = make_float2(mm, ll);
    }
  }
  if (n_split == 1) return;

  // the last CTA of this kv head to finish merges the splits
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&tickets[g], 1) == n_split - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // split weights: warp h' takes head h', lane l the splits l and l + 32 (at most 40 splits)
  static_assert(kDecMaxSplits <= 64, "two splits per lane");
  for (int h = warp; h < G; h += kDecWarps) {
    float2 a = make_float2(-INFINITY, 0.0f), b = make_float2(-INFINITY, 0.0f);
    if (lane < n_split) a = ld_cg(&part_ml[((size_t)g * n_split + lane) * G + h]);
    if (lane + 32 < n_split) b = ld_cg(&part_ml[((size_t)g * n_split + lane + 32) * G + h]);
    float mm = fmaxf(a.x, b.x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
    const float wa = a.x == -INFINITY ? 0.0f : exp2f(a.x - mm);
    const float wb = b.x == -INFINITY ? 0.0f : exp2f(b.x - mm);
    float ll = fmaf(wa, a.y, wb * b.y);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, off);
    const float inv = 1.0f / ll;
    if (lane < n_split) s_w[lane][h] = wa * inv;
    if (lane + 32 < n_split) s_w[lane + 32][h] = wb * inv;
  }
  __syncthreads();
  // outputs in float4 groups: kSub threads per group take every kSub-th split, all their loads
  // issued before the sums; the sub-sums of a group sit in adjacent lanes
  constexpr int kGroups = kOut / 4;
  constexpr int kSub = kGroups >= kDecThreads ? 1 : (2 * kGroups >= kDecThreads ? 2 : 4);
  constexpr int kPer = 20 / kSub;  // loads in flight per thread
  for (int t = threadIdx.x; t < kSub * kGroups; t += kDecThreads) {
    const int grp = t / kSub, par = t % kSub;
    const int h = (grp * 4) / D;
    const float4* base = reinterpret_cast<const float4*>(part_o + (size_t)g * n_split * kOut) + grp;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = par; s0 < n_split; s0 += kSub * kPer) {
      float4 t4[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u)
        if (s0 + kSub * u < n_split) t4[u] = ld_cg(base + (size_t)(s0 + kSub * u) * kGroups);
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int sp = s0 + kSub * u;
        if (sp < n_split) {
          const float w = s_w[sp][h];
          acc.x = fmaf(w, t4[u].x, acc.x);
          acc.y = fmaf(w, t4[u].y, acc.y);
          acc.z = fmaf(w, t4[u].z, acc.z);
          acc.w = fmaf(w, t4[u].w, acc.w);
        }
      }
    }
#pragma unroll
    for (int off = 1; off < kSub; off <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (par == 0) {
      uint2 pk = make_uint2(pack2(acc.x, acc.y), pack2(acc.z, acc.w));
      *reinterpret_cast<uint2*>(out + ((size_t)g * G * D + grp * 4) * 2) = pk;
    }
  }
  if (threadIdx.x == 0) tickets[g] = 0;  // ready for the next call
}

template <int D, int G>
cudaError_t launch_decode_t(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hkv, float scale,
                            void* out, const DecodeScratch& ws, cudaStream_t s) {
  // splits: about two CTAs per SM over all kv heads, at least 64 keys each, every one non-empty
  int splits = (ws.target_ctas + hkv - 1) / hkv;
  splits = splits < kDecMaxSplits ? splits : kDecMaxSplits;
  const int by_len = (n_keys + 63) / 64;
  splits = splits < by_len ? splits : by_len;
  if (splits < 1) splits = 1;
  const int per = (n_keys + splits - 1) / splits;
  splits = (n_keys + per - 1) / per;
  const float qscale = scale * 1.4426950408889634f;
  return launch_pdl(decode_attention_kernel<D, G>, dim3(splits, hkv), dim3(kDecThreads), 0, s,
                    (const uint8_t*)q, (const uint8_t*)k, (const uint8_t*)v, n_keys, hkv, per, qscale, ws.part_o,
                    ws.part_ml, ws.tickets, (uint8_t*)out);
}

template <int D>
cudaError_t launch_decode_d(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq, int32_t hkv,
                            float scale, void* out, const DecodeScratch& ws, cudaStream_t s) {
  switch (hq / hkv) {
    case 1: return launch_decode_t<D, 1>(q, k, v, n_keys, hkv, scale, out, ws, s);
    case 2: return launch_decode_t<D, 2>(q, k, v, n_keys, hkv, scale, out, ws, s);
    case 4: return launch_decode_t<D, 4>(q, k, v, n_keys, hkv, scale, out, ws, s);
    case 8: return launch_decode_t<D, 8>(q, k, v, n_keys, hkv, scale, out, ws, s);
    case 16: return launch_decode_t<D, 16>(q, k, v, n_keys, hkv, scale, out, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int32_t decode_max_splits() { return kDecMaxSplits; }

cudaError_t launch_decode_attention(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq,
                                    int32_t hkv, int32_t head_dim, float scale, void* out, const DecodeScratch& ws,
                                    cudaStream_t s) {
  if (n_keys <= 0) return cudaSuccess;
  if (head_dim == 128) return launch_decode_d<128>(q, k, v, n_keys, hq, hkv, scale, out, ws, s);
  if (head_dim == 64) return launch_decode_d<64>(q, k, v, n_keys, hq, hkv, scale, out, ws, s);
  return cudaErrorInvalidValue;
}

}  // namespace cb
