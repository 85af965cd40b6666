// Decode attention on the tensor cores ("rag的kvcache问题" §阶段 2 (Decode): the newest token is
// the only query; its [1, d] row meets the whole cached K/V, so the step is memory-bound):
//
//   out[h] = sum_{j < n_keys} softmax_j(scale q[h] . k[j, g]) v[j, g],  g = h / G.
//
// On the CUDA cores one key of one kv head costs about 2,000 flops of dot products, shuffle
// reductions and P V sums at G = 4-8, which an earlier form of this kernel found near the issue
// limit instead of the HBM limit (Llama-70B shape 23 us per layer, 0.22 of HBM). Here the G query
// heads of a kv head are rows 0 .. G-1 of a 128-row Q tile and each key tile takes the attention
// kernel's path: S = Q K_j^T (tcgen05, M 128, N 128 keys, K = D), one thread per head row turns S
// into P = 2^(s - m) in TMEM, and O += P V_j (P from TMEM, V MN-major). The tensor core does 16x
// the needed rows, which still leaves it idle most of the time: a 128-key tile is 64 KiB of K and
// V, about 2,850 cycles of an SM's share of HBM, against ~2,000 cycles of MMAs.
//
// Grid (splits, Hkv), one CTA per SM, splits x Hkv at most one wave: a CTA takes a contiguous
// range of key tiles of one kv head, and its first tiles are prefetched into L2 before it waits
// for the kernels it depends on. Warp 0 streams K and V tiles through two 3-stage rings (TMA,
// 128-byte swizzle), warp 1 issues the MMAs (S double-buffered in TMEM, so S_{j+1} is computed
// while the softmax works on tile j), warp 4 (TMEM lanes 0-31) runs the online softmax with one
// thread per head row (rows G .. 31 are inactive). Each CTA leaves (max, sum,
// unnormalised O rows) in the plan's decode scratch and the last CTA of a kv head (a ticket
// counter) merges the splits. Every mbarrier wait is bounded (2 s): a wait that gives up
// records a timeout, the CTA drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "attn_common.cuh"
#include "tc_common.cuh"
#include "tmem_ops.cuh"

namespace cb {
namespace {

constexpr int kTBM = 128;      // rows of the Q tile (the G head rows, the rest unused)
constexpr int kTBN = 128;      // keys per tile
constexpr int kTStages = 3;    // depth of the K and V rings
constexpr int kTThreads = 256;
constexpr int kWarpLoad = 0, kWarpMma = 1, kWarpSoftmax = 4;
constexpr uint32_t kTCols = 512;  // S buffers at 0 and 128, O at 256
constexpr float kTRescale = 8.0f;  // log2 units: O is rescaled only when a row's max grows by > 2^8
constexpr int kTMaxG = 32;         // head rows: the lanes of the softmax warp
constexpr int kTMaxSplits = 40;    // the plan's decode scratch holds 40 splits per kv head

struct TcBars {
  uint64_t q_full;
  uint64_t k_full[kTStages];
  uint64_t v_full[kTStages];
  uint64_t k_free[kTStages];  // S of the stage's tile complete (MMA commit)
  uint64_t pv_done[kTStages];  // P V of the stage's tile complete: V stage free, O updated (MMA commit)
  uint64_t s_done[2];          // S_j in TMEM buffer j % 2 (MMA commit)
  uint64_t p_ready[2];         // P_j written over S_j (softmax warp)
  uint64_t drain;
};

struct TcParams {
  int n_keys;
  int G;  // query heads per kv head
  int tiles_per_split;
  int n_tiles;      // key tiles in all
  float scale_log2;
  float* part_o;
  float2* part_ml;
  int32_t* tickets;
  uint8_t* out;
  int32_t* err;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// PROBE: the wait-timeout probe (test support only): the producer arms key tile 1's barrier of
// every CTA but never copies the tile, and every wait gives up after kProbeTimeoutNs, so each CTA
// that has a second tile takes its failure path (timeout recorded, copies and tensor-core work
// drained, TMEM freed; the ticket is still taken, so the counters stay consistent).
template <int D, bool PROBE = false>
__global__ void __launch_bounds__(kTThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kQBox = kTBM * 128;  // one 64-column box of the Q tile
  constexpr uint32_t kKVBox = kTBN * 128;
  constexpr uint32_t kQBytes = kBoxes * kQBox;
  constexpr uint32_t kKVBytes = kBoxes * kKVBox;
  constexpr uint32_t kColO = 256;
  constexpr uint64_t kLimit = PROBE ? kProbeTimeoutNs : kTimeoutNs;

  extern __shared__ uint8_t smem_raw[];
  __shared__ TcBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_last;

  pdl_launch_dependents();
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK0 = sQ + kQBytes;
  const uint32_t sV0 = sK0 + kTStages * kKVBytes;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = blockIdx.y, split = blockIdx.x, n_split = gridDim.x;
  const int j0 = split * p.tiles_per_split;  // first key tile of this CTA
  const int n = min(p.tiles_per_split, p.n_tiles - j0);  // its tiles (>= 1 by the launch)

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.k_free[s]), 1);
      mbar_init(smem_u32(&bars.pv_done[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars.s_done[b]), 1);
      mbar_init(smem_u32(&bars.p_ready[b]), 1);
    }
    mbar_init(smem_u32(&bars.drain), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else if (warp == 2 && lane == 0) {
    // While the kernels before this one finish: the tensor maps, and this CTA's first K and V
    // tiles into L2 (a prefetch only fills L2, so it cannot make a later load read stale data).
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_q) : "memory");
    for (int j = 0; j < n && j < kTStages; ++j)
#pragma unroll
      for (int b = 0; b < kBoxes; ++b) {
        asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(&tm_k), "r"(b * 64),
                     "r"(g), "r"((j0 + j) * kTBN)
                     : "memory");
        asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(&tm_v), "r"(b * 64),
                     "r"(g), "r"((j0 + j) * kTBN)
                     : "memory");
      }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  pdl_wait();  // q, k and v come from the kernels before this one

  if (warp == kWarpLoad) {
    if (lane == 0) {
      const uint32_t qb = smem_u32(&bars.q_full);
      mbar_expect_tx(qb, (uint32_t)(kBoxes * p.G * 128));  // G rows of each box
#pragma unroll
      for (int b = 0; b < kBoxes; ++b) tma_load_3d(sQ + b * kQBox, &tm_q, qb, b * 64, g * p.G, 0);
      int nk = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % kTStages;
        if (j >= kTStages) {
          const uint32_t par = ((j / kTStages) - 1) & 1;
          if (!mbar_spin(smem_u32(&bars.k_free[st]), par, abort_flag, p.err, 60, kLimit)) break;
          if (!mbar_spin(smem_u32(&bars.pv_done[st]), par, abort_flag, p.err, 61, kLimit)) break;
        }
        const int key0 = (j0 + j) * kTBN;  // past n_keys: zero fill
        const uint32_t kb = smem_u32(&bars.k_full[st]), vb = smem_u32(&bars.v_full[st]);
        mbar_expect_tx(kb, kKVBytes);
        if (!(PROBE && j == 1)) {  // the probe never copies key tile 1: its barrier cannot complete
#pragma unroll
          for (int b = 0; b < kBoxes; ++b)
            tma_load_3d(sK0 + st * kKVBytes + b * kKVBox, &tm_k, kb, b * 64, g, key0);
        }
        mbar_expect_tx(vb, kKVBytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) tma_load_3d(sV0 + st * kKVBytes + b * kKVBox, &tm_v, vb, b * 64, g, key0);
        nk = j + 1;
      }
      // every copy issued has landed before the CTA may exit
      mbar_wait(qb, 0, abort_flag, p.err, 62, false, kLimit);
      for (int j = nk - kTStages < 0 ? 0 : nk - kTStages; j < nk; ++j) {
        mbar_wait(smem_u32(&bars.k_full[j % kTStages]), (j / kTStages) & 1, abort_flag, p.err, 63, false, kLimit);
        mbar_wait(smem_u32(&bars.v_full[j % kTStages]), (j / kTStages) & 1, abort_flag, p.err, 64, false, kLimit);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    constexpr uint32_t idesc_s = idesc_bf16(kTBM, kTBN, false);
    constexpr uint32_t idesc_o = idesc_bf16(kTBM, D, true);
    const uint64_t dq = sdesc(sQ, 16, 1024);
    const uint64_t dk0 = sdesc(sK0, 16, 1024);
    const uint64_t dv0 = sdesc(sV0, kKVBox, 1024);
    auto spin_all = [&](uint32_t bar, uint32_t parity, int site) -> bool {
      return __all_sync(0xffffffffu, mbar_spin(bar, parity, abort_flag, p.err, site, kLimit));
    };
    // S_j = Q K_j^T into buffer j % 2; its commit frees the K stage and hands S_j to the softmax.
    auto issue_s = [&](int j) -> bool {
      const int st = j % kTStages, b = j & 1;
      if (!spin_all(smem_u32(&bars.k_full[st]), (j / kTStages) & 1, 65)) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dk = dk0 + (uint64_t)((st * kKVBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int bx = ks / 4, kk = ks % 4;
          mma_ss(tmem + (uint32_t)(b * kTBN), dq + (uint64_t)((bx * kQBox + kk * 32) >> 4),
                 dk + (uint64_t)((bx * kKVBox + kk * 32) >> 4), idesc_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&bars.k_free[st]));
        tc_commit(smem_u32(&bars.s_done[b]));
      }
      __syncwarp();
      return true;
    };
    bool ok = spin_all(smem_u32(&bars.q_full), 0, 66) && issue_s(0) && (n < 2 || issue_s(1));
    for (int j = 0; j < n && ok; ++j) {
      // O += P_j V_j once the softmax has written P_j and V_j is in; then S_{j+2} into the same
      // buffer (executed after this P V, which reads P_j from it).
      const int b = j & 1, st = j % kTStages;
      ok = spin_all(smem_u32(&bars.p_ready[b]), (j >> 1) & 1, 67) &&
           spin_all(smem_u32(&bars.v_full[st]), (j / kTStages) & 1, 68);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dv = dv0 + (uint64_t)((st * kKVBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kTBN / 16; ++ks)
          mma_ts(tmem + kColO, tmem + (uint32_t)(b * kTBN) + ks * 8, dv + (uint64_t)((ks * 16 * 128) >> 4), idesc_o,
                 (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(smem_u32(&bars.pv_done[st]));
      }
      __syncwarp();
      if (j + 2 < n) ok = issue_s(j + 2);
    }
    // every MMA issued here completes before TMEM is freed
    if (elect_one()) tc_commit(smem_u32(&bars.drain));
    __syncwarp();
    mbar_wait(smem_u32(&bars.drain), 0, abort_flag, p.err, 69, false, kLimit);
  }

  // Softmax (warp 4, one thread per head row) and the CTA's partial result.
  float m_ref = -INFINITY, l = 0.0f;  // row max (log2 units) that O and l are scaled to, row sum
  bool ok = true;
  const bool row = lane < p.G;
  const uint32_t lanes = tmem;  // warp 4 reads TMEM lanes 0-31
  if (warp == kWarpSoftmax) {
    auto wait_all = [&](uint32_t bar, uint32_t parity, int site) -> bool {
      return __all_sync(0xffffffffu, mbar_spin(bar, parity, abort_flag, p.err, site, kLimit));
    };
    for (int j = 0; j < n && ok; ++j) {
      const int b = j & 1;
      ok = wait_all(smem_u32(&bars.s_done[b]), (j >> 1) & 1, 70);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[kTBN];
#pragma unroll
      for (int c = 0; c < kTBN; c += 32)
        tmem_ld_x32_async(lanes + (uint32_t)(b * kTBN + c), *reinterpret_cast<uint32_t(*)[32]>(&sv[c]));
      // one wait per chunk, so that no use of a chunk's registers moves above the wait
#pragma unroll
      for (int c = 0; c < kTBN; c += 32) tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&sv[c]));
      // keys past n_keys (the zero-filled end of the last tile) and inactive rows get -inf
      const int lim = row ? p.n_keys - 1 - (j0 + j) * kTBN : -1;
      if (lim < kTBN - 1) {
#pragma unroll
        for (int c = 0; c < kTBN; ++c)
          if (c > lim) sv[c] = 0xff800000u;
      }
      float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kTBN; c += 8) {
        tm[0] = max3(tm[0], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
        tm[1] = max3(tm[1], __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
        tm[2] = max3(tm[2], __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
        tm[3] = max3(tm[3], __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
      }
      const float mt = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])) * p.scale_log2;  // -inf: no key
      const bool up = mt > m_ref + kTRescale;  // always at a row's first tile
      if (__any_sync(0xffffffffu, up)) {
        const float alpha = up ? ex2(m_ref - mt) : 1.0f;  // 0 while the row had nothing
        const bool scale_o = up && m_ref != -INFINITY;
        if (up) {
          l *= alpha;
          m_ref = mt;
        }
        // O holds the sum through tile j - 1: wait for that P V, then scale it
        if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
          ok = wait_all(smem_u32(&bars.pv_done[(j - 1) % kTStages]), ((j - 1) / kTStages) & 1, 71);
          if (!ok) break;
          tc_fence_after();
          const float a = scale_o ? alpha : 1.0f;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld_x32(lanes + kColO + c0, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
            tmem_st_x32(lanes + kColO + c0, o);
          }
          tmem_st_wait();
        }
      }
      // P = 2^(s * scale - m_ref) <= 2^8 as bf16 pairs over the first 64 columns of S_j, and its sum
      const float neg_m = m_ref == -INFINITY ? 0.0f : -m_ref;
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(neg_m, neg_m);
      uint64_t ps2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) ps2[q] = f2_pack(0.0f, 0.0f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int c = h * 64 + 2 * e;
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nm2), t0, t1);
          const float p0 = ex2(t0), p1 = ex2(t1);
          ps2[e & 3] = f2_add(ps2[e & 3], f2_pack(p0, p1));
          pk[e] = pack2(p0, p1);
        }
        tmem_st_x32(lanes + (uint32_t)(b * kTBN + h * 32), pk);
      }
      float sa, sb;
      f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), sa, sb);
      l += sa + sb;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.p_ready[b]));
    }
    if (ok) ok = wait_all(smem_u32(&bars.pv_done[(n - 1) % kTStages]), ((n - 1) / kTStages) & 1, 72);
    if (ok) {
      tc_fence_after();
      const size_t unit = (size_t)g * n_split + split;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld_x32(lanes + kColO + c0, o);
        if (row) {
          if (n_split == 1) {
            const float inv = 1.0f / l;
            float f[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * inv;
            uint8_t* dst = p.out + ((size_t)(g * p.G + lane) * D + c0) * 2;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) *reinterpret_cast<uint4*>(dst + q4 * 16) = pack8(f + q4 * 8);
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + ((unit * p.G + lane) * D + c0));
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                                    __uint_as_float(o[4 * q4 + 2]), __uint_as_float(o[4 * q4 + 3]));
          }
        }
      }
      if (row && n_split > 1) p.part_ml[unit * p.G + lane] = make_float2(m_ref, l);
    }
    if (!__all_sync(0xffffffffu, ok)) *abort_flag = 1;
  }

  // The last CTA of this kv head to finish merges the splits.
  tc_fence_before();
  __syncthreads();
  // Every CTA takes its ticket, also one whose wait gave up (its partial is then missing, the
  // error word says so), so the counter always completes and is reset for the next call.
  const bool merged = n_split > 1;
  if (merged) {
    __threadfence();
    if (threadIdx.x == 0) s_last = atomicAdd(&p.tickets[g], 1) == n_split - 1;
  }
  __syncthreads();
  if (merged && s_last) {
    __threadfence();
    // The partial O rows of this thread's first output group go out first, so that their round trip
    // to L2 overlaps the one of the weights below (up to kMergeBatch splits per batch of loads).
    constexpr int kMergeBatch = 8;
    const int n_groups = p.G * D / 4;
    const float4* src = reinterpret_cast<const float4*>(p.part_o + (size_t)g * n_split * p.G * D);
    float4 first[kMergeBatch];
    if ((int)threadIdx.x < n_groups) {
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u)
        if (u < n_split) first[u] = __ldcg(src + (size_t)u * n_groups + threadIdx.x);
    }
    // merge weights [split][head] in the K ring, free now (every load landed, every MMA completed)
    float(*s_w)[kTMaxG] = reinterpret_cast<float(*)[kTMaxG]>(smem_raw + (sK0 - smem_u32(smem_raw)));
    // weights: warp w takes heads w, w + 8, ...; lane l the splits l and l + 32
    for (int h = warp; h < p.G; h += kTThreads / 32) {
      float2 a = make_float2(-INFINITY, 0.0f), c = make_float2(-INFINITY, 0.0f);
      if (lane < n_split) a = __ldcg(&p.part_ml[((size_t)g * n_split + lane) * p.G + h]);
      if (lane + 32 < n_split) c = __ldcg(&p.part_ml[((size_t)g * n_split + lane + 32) * p.G + h]);
      float mm = fmaxf(a.x, c.x);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
      const float wa = a.x == -INFINITY ? 0.0f : exp2f(a.x - mm);
      const float wc = c.x == -INFINITY ? 0.0f : exp2f(c.x - mm);
      float ll = fmaf(wa, a.y, wc * c.y);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, off);
      const float inv = 1.0f / ll;
      if (lane < n_split) s_w[lane][h] = wa * inv;
      if (lane + 32 < n_split) s_w[lane + 32][h] = wc * inv;
    }
    __syncthreads();
    // outputs in float4 groups, each thread summing the splits of its groups with a batch of loads
    // in flight at a time
    for (int grp = threadIdx.x; grp < n_groups; grp += kTThreads) {
      const int h = (grp * 4) / D;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < n_split; s0 += kMergeBatch) {
        float4 t4[kMergeBatch];
        if (s0 == 0 && grp == (int)threadIdx.x) {
#pragma unroll
          for (int u = 0; u < kMergeBatch; ++u) t4[u] = first[u];
        } else {
#pragma unroll
          for (int u = 0; u < kMergeBatch; ++u)
            if (s0 + u < n_split) t4[u] = __ldcg(src + (size_t)(s0 + u) * n_groups + grp);
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          if (s0 + u < n_split) {
            const float w = s_w[s0 + u][h];
            acc.x = fmaf(w, t4[u].x, acc.x);
            acc.y = fmaf(w, t4[u].y, acc.y);
            acc.z = fmaf(w, t4[u].z, acc.z);
            acc.w = fmaf(w, t4[u].w, acc.w);
          }
        }
      }
      const uint2 pk = make_uint2(pack2(acc.x, acc.y), pack2(acc.z, acc.w));
      *reinterpret_cast<uint2*>(p.out + ((size_t)g * p.G * D + grp * 4) * 2) = pk;
    }
    if (threadIdx.x == 0) p.tickets[g] = 0;  // ready for the next call
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTCols) : "memory");
  }
}

template <int D, bool PROBE = false>
cudaError_t launch_decode_tc_t(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq, int32_t hkv,
                               float scale, void* out, const DecodeScratch& ws, int32_t* err, cudaStream_t s) {
  const int G = hq / hkv;
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hq, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hq * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, 1};
    if (!encode_map(&tq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)n_keys};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTBN};
    if (!encode_map(&tk, k, 3, dims, strides, box) || !encode_map(&tv, v, 3, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  const int n_tiles = (n_keys + kTBN - 1) / kTBN;
  const int sms = ws.sms > 0 ? ws.sms : 1;
  int max_splits = sms / hkv;
  if (max_splits > kTMaxSplits) max_splits = kTMaxSplits;
  if (max_splits < 1) max_splits = 1;
  const int per = (n_tiles + max_splits - 1) / max_splits;
  const int splits = (n_tiles + per - 1) / per;  // every split has at least one tile
  TcParams p;
  p.n_keys = n_keys;
  p.G = G;
  p.tiles_per_split = per;
  p.n_tiles = n_tiles;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.part_o = ws.part_o;
  p.part_ml = ws.part_ml;
  p.tickets = ws.tickets;
  p.out = static_cast<uint8_t*>(out);
  p.err = err;
  const size_t smem = 1024 + (size_t)(D / 64) * (kTBM * 128 + 2 * kTStages * kTBN * 128);
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = set_smem_limit_once(decode_tc_kernel<D, PROBE>, (int)smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tc_kernel<D, PROBE>, dim3(splits, hkv), dim3(kTThreads), smem, s, tq, tk, tv, p);
}

}  // namespace

int32_t decode_max_splits() { return kTMaxSplits; }

bool decode_tc_supported(int32_t hq, int32_t hkv, int32_t head_dim) {
  return (head_dim == 64 || head_dim == 128) && hkv > 0 && hq % hkv == 0 && hq / hkv <= kTMaxG;
}

cudaError_t launch_decode_tc(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq, int32_t hkv,
                             int32_t head_dim, float scale, void* out, const DecodeScratch& ws, int32_t* err,
                             cudaStream_t s) {
  if (n_keys <= 0) return cudaErrorInvalidValue;
  if (head_dim == 128) return launch_decode_tc_t<128>(q, k, v, n_keys, hq, hkv, scale, out, ws, err, s);
  if (head_dim == 64) return launch_decode_tc_t<64>(q, k, v, n_keys, hq, hkv, scale, out, ws, err, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_timeout_probe(const void* q, const void* k, const void* v, int32_t n_keys, int32_t hq,
                                        int32_t hkv, float scale, void* out, const DecodeScratch& ws, int32_t* err,
                                        cudaStream_t s) {
  if (n_keys <= kTBN) return cudaErrorInvalidValue;  // no key tile 1 to miss
  return launch_decode_tc_t<128, true>(q, k, v, n_keys, hq, hkv, scale, out, ws, err, s);
}

}  // namespace cb
