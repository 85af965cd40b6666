// The step before the blend: the QKV projection of the rows a layer recomputes, on sm_103a
// tensor cores ("rag的kvcache问题" §阶段一: each token's q, k, v is its hidden vector times the
// projection weights, computed as one product of the stacked rows; §渐进式过滤机制: a layer
// recomputes only its candidate tokens and the query suffix).
//
//   y[i, :] = x[x_index[i], :] W^T,  W = W_qkv [(Hq + 2 Hkv) D, d_model] (one output feature per row)
//   q[t] = y[i, Q heads], k[t] = y[i, K heads], v[t] = y[i, V heads],  t = tokens[i],
// with q and k optionally RoPE-encoded at position t (the plan's cos/sin table) in the epilogue,
// all written token-indexed as bf16: the layout the blend reads its recomputed rows from.
//
// (x_index null: row i of x; tokens null: token i). With an index list the rows of X are first
// gathered into a contiguous workspace by a streaming kernel (2 m d_model bytes each way): a
// 128-byte-swizzled TMA tile must land on a 1024-byte boundary, which four-row gathers into one
// tile cannot all meet; without one the tiles read x in place. A cluster of two CTAs then computes a
// 256 x 256 output tile with tcgen05 cta_group::2: CTA r holds 128 gathered rows and W rows
// n0 + 128 r .. n0 + 128 r + 127 of the tile's 256 output features (two 128-wide heads or four
// 64-wide heads of one of Q, K, V), and the pair's MMA (M 256, N 256, K 16; bf16 in, fp32
// accumulate), issued by CTA 0, reads both CTAs' shared memory and leaves each CTA's 128 rows x
// 256 features in 256 columns of its own TMEM. Holding half of each W slice per SM makes a
// stage 32 KiB (128 x 64 of X and of W, 128-byte swizzled), so seven stages fit and cover the
// load latency, which four 48 KiB stages of a one-CTA 128 x 256 tile could not (its tensor pipe
// idled a quarter of the K loop). Warp 0 of each CTA issues its loads, which complete on CTA 0's
// "full" barrier (the cta_group::2 form of the tensor copy; CTA 0 expects the pair's bytes);
// warp 1 of CTA 0 issues the MMAs and commits each stage to both CTAs' "empty" barriers
// (multicast); both poll their barriers (a sleeping wait resumes hundreds of cycles late).
// TMEM allocation, barrier set-up and the first W slices' L2 prefetch happen before the wait
// on the kernels this one depends on. Then all eight warps of each CTA turn its accumulator
// into bf16 rows in the drained ring (one output row per thread; warps g and g + 4 read TMEM
// lanes 32 g .. 32 g + 31 and take half of the tile's heads each): the tile's cos/sin rows come
// in coalesced (one token row per warp instruction), the RoPE-encoded rows go out coalesced.
// Every mbarrier wait is bounded (2 s); a timeout records an error, the CTA drains its copies
// and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tmem_ops.cuh"

namespace cb {
namespace {

constexpr int kPM = 128;  // gathered rows per tile
constexpr int kPN = 256;  // output features per tile
constexpr int kPK = 64;   // K slice per stage (one 128-byte swizzle row of bf16)
constexpr int kPThreads = 256;
constexpr uint32_t kPTmemCols = 256;

struct ProjParams {
  const int32_t* tokens;  // token of output row i (null: token i)
  int m;
  int n_tokens;
  int d_model;
  int hq, hkv, head_dim;
  int encode;
  int style;
  const float2* tab;  // [n_tokens][head_dim / 2] (cos, sin)
  uint8_t* q;
  uint8_t* k;
  uint8_t* v;
  int32_t* err;
};

// Rows of X to a contiguous [m, d_model] buffer: one warp per row, 16-byte accesses, up to 8 KiB
// of a row's loads in flight before its stores; an index outside X gives a zero row and an error
// record.
__global__ void __launch_bounds__(256) gather_rows_kernel(uint8_t* dst, const uint8_t* src, const int32_t* rows,
                                                          int m, int n_src, int row_bytes, int32_t* err) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (warp >= m) return;
  const int t = rows[warp];
  uint8_t* d = dst + (size_t)warp * row_bytes;
  if (t < 0 || t >= n_src) {
    if (lane == 0) record_error(err, kErrIndex, warp);
    for (int c = lane * 16; c < row_bytes; c += 32 * 16) st_stream(d + c, make_uint4(0u, 0u, 0u, 0u));
    return;
  }
  const uint8_t* sp = src + (size_t)t * row_bytes;
  constexpr int B = 16;
  for (int c0 = lane * 16; c0 < row_bytes; c0 += 32 * 16 * B) {
    uint4 v[B];
#pragma unroll
    for (int b = 0; b < B; ++b)
      if (c0 + b * 512 < row_bytes) v[b] = ld_stream(sp + c0 + b * 512);
#pragma unroll
    for (int b = 0; b < B; ++b)
      if (c0 + b * 512 < row_bytes) st_stream(d + c0 + b * 512, v[b]);
  }
}

// Shared-memory accesses by 32-bit shared-window address, and the 16-byte global -> shared copy
// (cp.async, cached in L2 only) with its wait.
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_u4(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Named barrier of the two warps g and g + 4 of the epilogue (ids 1-4; 0 is __syncthreads).
__device__ __forceinline__ void pair_bar_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// Epilogue on all eight warps: warps g and g + 4 share TMEM lanes 32 g .. 32 g + 31 (the tile
// rows of group g) and split the tile's heads; a named barrier per pair orders their shared
// staging. Whether the accumulator is complete is decided for the whole CTA, so a wait that
// gave up in one warp cannot leave its partner at a pair barrier.
template <int D>
__device__ __forceinline__ void proj_epilogue(const ProjParams& p, uint32_t acc_bar, uint32_t tmem, uint32_t sA0,
                                              const int* s_rows, int m0, int n0, volatile int* abort_flag,
                                              uint64_t limit_ns) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool acc_ok = mbar_wait(acc_bar, 0, abort_flag, p.err, 44, true, limit_ns);
  if (__syncthreads_and(acc_ok ? 1 : 0)) {
    tc_fence_after();
    const int g = warp & 3, upper = warp >> 2;
    const int r = g * 32 + lane;
    const int half_rows = g * 32 + (upper ? 0 : 16);  // the 16 rows this warp loads and stores
    const uint32_t lane_base = tmem + ((uint32_t)(g * 32) << 16);
    // Every MMA has completed, so the ring is free: it stages the tile's cos/sin rows (loaded
    // coalesced, one token row per warp instruction) and the bf16 output rows (stored
    // coalesced, one tile row per warp instruction). Row pitches are 16 bytes past a multiple
    // of 128, so a thread per row touches every bank once per 16-byte step.
    constexpr uint32_t kOutPitch = kPN * 2 + 16;
    constexpr uint32_t kTabPitch = D * 4 + 16;  // D / 2 (cos, sin) pairs
    const uint32_t out_s = sA0;
    const uint32_t tab_s = sA0 + kPM * kOutPitch;
    const int n_qk = (p.hq + p.hkv) * D;  // features that RoPE encodes
    const bool rope_tile = p.encode != 0 && n0 < n_qk;
    if (rope_tile) {
      for (int i = 0; i < 16; ++i) {
        const int t = s_rows[half_rows + i];
        if (t >= 0 && lane * 16 < D * 4)
          cp_async16(tab_s + (uint32_t)(half_rows + i) * kTabPitch + lane * 16,
                     reinterpret_cast<const uint8_t*>(p.tab + (size_t)t * (D / 2)) + lane * 16);
      }
      cp_async_wait_all();
    }
    pair_bar_sync(1 + g);
    const uint32_t my_out = out_s + (uint32_t)r * kOutPitch;
    const uint32_t my_tab = tab_s + (uint32_t)r * kTabPitch;
    constexpr int kHeads = kPN / D;
#pragma unroll 1
    for (int hh = upper ? 0 : kHeads / 2; hh < (upper ? kHeads / 2 : kHeads); ++hh) {
      const int f0 = n0 + hh * D;  // first output feature of this head
      // warp-uniform (tcgen05.ld is a whole-warp instruction): a row without a token computes
      // from unloaded table entries and is never stored
      const bool rope = rope_tile && f0 < n_qk;
      const uint32_t col = lane_base + hh * D;
      if (rope && p.style == 0) {
        // pairs (j, j + D/2): columns j0.. and D/2 + j0.. of the head
#pragma unroll 1
        for (int j0 = 0; j0 < D / 2; j0 += 32) {
          uint32_t a[32], b[32];
          tmem_ld_x32_async(col + j0, a);
          tmem_ld_x32_async(col + D / 2 + j0, b);
          tmem_wait_ld(a);
          tmem_wait_ld(b);
          float oa[32], ob[32];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const float4 c = lds_f4(my_tab + (uint32_t)(j0 + 2 * e2) * 8);  // pairs j0 + 2 e2, + 1
            const float x0 = __uint_as_float(a[2 * e2]), y0 = __uint_as_float(b[2 * e2]);
            const float x1 = __uint_as_float(a[2 * e2 + 1]), y1 = __uint_as_float(b[2 * e2 + 1]);
            oa[2 * e2] = x0 * c.x - y0 * c.y;
            ob[2 * e2] = x0 * c.y + y0 * c.x;
            oa[2 * e2 + 1] = x1 * c.z - y1 * c.w;
            ob[2 * e2 + 1] = x1 * c.w + y1 * c.z;
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            sts_u4(my_out + (uint32_t)(hh * D + j0 + q4 * 8) * 2, pack8(oa + q4 * 8));
            sts_u4(my_out + (uint32_t)(hh * D + D / 2 + j0 + q4 * 8) * 2, pack8(ob + q4 * 8));
          }
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t a[32];
          tmem_ld_x32(col + c0, a);
          float o[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(a[e]);
          if (rope) {  // pairs (2j, 2j + 1)
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) {
              const float4 c = lds_f4(my_tab + (uint32_t)(c0 / 2 + 2 * e2) * 8);
              const float x0 = o[4 * e2], y0 = o[4 * e2 + 1], x1 = o[4 * e2 + 2], y1 = o[4 * e2 + 3];
              o[4 * e2] = x0 * c.x - y0 * c.y;
              o[4 * e2 + 1] = x0 * c.y + y0 * c.x;
              o[4 * e2 + 2] = x1 * c.z - y1 * c.w;
              o[4 * e2 + 3] = x1 * c.w + y1 * c.z;
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) sts_u4(my_out + (uint32_t)(hh * D + c0 + q4 * 8) * 2, pack8(o + q4 * 8));
        }
      }
    }
    pair_bar_sync(1 + g);
    // Coalesced stores of this warp's 16 rows: lane l takes tile features 8 l .. 8 l + 7.
    const int f = n0 + lane * 8;
    const int n_out = (p.hq + 2 * p.hkv) * D;
    uint8_t* dst_base = nullptr;
    int heads_in = 0, head = 0;
    if (f < p.hq * D) {
      dst_base = p.q; heads_in = p.hq; head = f / D;
    } else if (f < n_qk) {
      dst_base = p.k; heads_in = p.hkv; head = f / D - p.hq;
    } else if (f < n_out) {
      dst_base = p.v; heads_in = p.hkv; head = f / D - p.hq - p.hkv;
    }
    const size_t col_bytes = (size_t)head * D * 2 + (size_t)(f % D) * 2;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int row = half_rows + i;
      const int ti = s_rows[row];
      if (m0 + row < p.m && ti >= 0 && dst_base != nullptr) {
        const uint4 val = lds_u4(out_s + (uint32_t)row * kOutPitch + lane * 16);
        *reinterpret_cast<uint4*>(dst_base + (size_t)ti * heads_in * D * 2 + col_bytes) = val;
      }
    }
  }
}

// ---- CTA-pair kernel ----
constexpr int kQStages = 7;
constexpr uint32_t kQHalfBytes = kPM * kPK * 2;  // 16 KiB: 128 rows x 64 of A, or of half of B

struct PairBars {
  uint64_t full[kQStages];   // CTA 0: both CTAs' A rows and W halves of the stage landed
  uint64_t empty[kQStages];  // the pair's MMAs of the stage completed
  uint64_t acc_full;             // every MMA completed
  uint64_t drain;                // CTA 0's MMA issue loop ended and its MMAs completed
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_smem(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Tensor copy into this CTA's shared memory whose completion is counted on `bar_cluster`, a
// barrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void mma_ss_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive on the barrier at this shared-memory offset in both CTAs of the pair once every MMA this
// thread issued so far has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// PROBE: the wait-timeout probe (test support only): CTA 0 arms the barrier of K step 1 for the
// pair's bytes but never copies its own share, and every wait gives up after kProbeTimeoutNs, so
// both CTAs of every pair take the failure path (timeout recorded, the MMAs issued so far drained,
// TMEM freed, both at the final cluster barrier).
template <int D, bool PROBE = false>
__global__ void __launch_bounds__(kPThreads, 1)
    qkv_projection_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                               const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ PairBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_rows[kPM];

  pdl_launch_dependents();
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair's MMAs
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + kQStages * kQHalfBytes;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m0 = blockIdx.x * kPM;          // this CTA's rows
  const int n0 = blockIdx.y * kPN;          // the pair's 256 output features
  const int nb = n0 + (int)rank * (kPN / 2);  // this CTA's half of the W slice
  const int n_k = p.d_model / kPK;
  constexpr uint64_t kLimit = PROBE ? kProbeTimeoutNs : kTimeoutNs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(smem_u32(&bars.full[s]), 1);  // used in CTA 0: its producer's expect_tx
      mbar_init(smem_u32(&bars.empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.acc_full), 1);
    mbar_init(smem_u32(&bars.drain), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {  // one warp of each CTA allocates the pair's columns together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kPTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else if (threadIdx.x == 32) {
    // While the kernels before this one finish: the tensor maps, and this CTA's first W slices
    // into L2 (a prefetch only fills L2, so it cannot make a later load read stale data).
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_x) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_w) : "memory");
    for (int kk = 0; kk < kQStages && kk < n_k; ++kk)
      asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(&tm_w), "r"(kk * kPK), "r"(nb)
                   : "memory");
  }
  // both CTAs' barriers initialised and TMEM allocated before any commit or MMA of the pair
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  pdl_wait();  // the rows and hidden states come from the kernels before this one

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full0 = peer_smem(smem_u32(&bars.full[0]), 0);  // CTA 0's barriers
      int issued = 0;
      for (int kk = 0; kk < n_k; ++kk) {
        const int st = kk % kQStages;
        if (kk >= kQStages &&
            !mbar_spin(smem_u32(&bars.empty[st]), ((kk / kQStages) - 1) & 1, abort_flag, p.err, 50, kLimit))
          break;
        if (rank == 0) mbar_expect_tx(smem_u32(&bars.full[st]), 4 * kQHalfBytes);  // both CTAs' bytes
        const uint32_t fb = full0 + (uint32_t)st * 8u;
        issued = kk + 1;
        if (PROBE && rank == 0 && kk == 1) continue;  // the probe's stage that can never complete
        tma_load_2d_pair(sA0 + st * kQHalfBytes, &tm_x, fb, kk * kPK, m0);  // rows past m read as zeros
        tma_load_2d_pair(sB0 + st * kQHalfBytes, &tm_w, fb, kk * kPK, nb);
      }
      // CTA 0: every copy of the pair that was issued has landed (CTA 1 waits for CTA 0 at the
      // final cluster barrier, so it cannot exit with copies in flight either)
      if (rank == 0)
        for (int kk = issued - kQStages < 0 ? 0 : issued - kQStages; kk < issued; ++kk)
          mbar_wait(smem_u32(&bars.full[kk % kQStages]), (kk / kQStages) & 1, abort_flag, p.err, 51, false, kLimit);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) {
      constexpr uint32_t idesc = idesc_bf16(2 * kPM, kPN, false);
      const uint64_t da0 = sdesc(sA0, 16, 1024);
      const uint64_t db0 = sdesc(sB0, 16, 1024);
      bool ok = true;
      for (int kk = 0; kk < n_k && ok; ++kk) {
        const int st = kk % kQStages;
        const uint32_t par = (kk / kQStages) & 1;
        ok = __all_sync(0xffffffffu, mbar_spin(smem_u32(&bars.full[st]), par, abort_flag, p.err, 52, kLimit));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t da = da0 + (uint64_t)((st * kQHalfBytes) >> 4);
          const uint64_t db = db0 + (uint64_t)((st * kQHalfBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < kPK / 16; ++ks)
            mma_ss_pair(tmem, da + (uint64_t)((ks * 32) >> 4), db + (uint64_t)((ks * 32) >> 4), idesc,
                        (kk > 0 || ks > 0) ? 1u : 0u);
          tc_commit_pair(smem_u32(&bars.empty[st]));
          if (kk == n_k - 1) tc_commit_pair(smem_u32(&bars.acc_full));
        }
        __syncwarp();
      }
      if (elect_one()) tc_commit_pair(smem_u32(&bars.drain));
      __syncwarp();
    }
    // neither CTA frees TMEM or exits while the pair's MMAs may still read or write it
    mbar_wait(smem_u32(&bars.drain), 0, abort_flag, p.err, 54, false, kLimit);
  } else if (warp >= 4) {
    // token of each of this CTA's rows (-1: past m, or outside the cache: not stored); only the
    // epilogue reads them, after its CTA-wide barrier
    const int i = m0 + (int)threadIdx.x - 128;
    int t = -1;
    if (i < p.m) {
      t = p.tokens ? p.tokens[i] : i;
      if (t < 0 || t >= p.n_tokens) {
        if (blockIdx.y == 0) record_error(p.err, kErrIndex, i);  // once per row
        t = -1;
      }
    }
    s_rows[threadIdx.x - 128] = t;
  }

  proj_epilogue<D>(p, smem_u32(&bars.acc_full), tmem, sA0, s_rows, m0, n0, abort_flag, kLimit);

  tc_fence_before();
  cluster_sync_all();  // neither CTA exits while the other may still arrive on its barriers
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPTmemCols) : "memory");
  }
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (enc == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool PROBE = false>
cudaError_t launch_proj_pair(const ProjParams& p, const void* x, const void* w, cudaStream_t s) {
  const int n_out = (p.hq + 2 * p.hkv) * D;
  CUtensorMap tx, tw;
  if (!encode_2d(&tx, x, (uint64_t)p.d_model, (uint64_t)p.m, kPK, kPM) ||
      !encode_2d(&tw, w, (uint64_t)p.d_model, (uint64_t)n_out, kPK, kPN / 2))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)kQStages * 2 * kQHalfBytes;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = set_smem_limit_once(qkv_projection_pair_kernel<D, PROBE>, (int)smem, configured);
  if (e != cudaSuccess) return e;
  const int m_tiles = (p.m + kPM - 1) / kPM;
  const dim3 grid((unsigned)(2 * ((m_tiles + 1) / 2)), (n_out + kPN - 1) / kPN);  // whole pairs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, qkv_projection_pair_kernel<D, PROBE>, tx, tw, p);
}

}  // namespace

cudaError_t launch_qkv_projection(const void* x, int32_t x_rows, int32_t d_model, const int32_t* x_index,
                                  const int32_t* tokens, int32_t m, void* x_gathered, const void* w, int32_t n_tokens,
                                  int32_t hq, int32_t hkv, int32_t head_dim, int32_t encode, int32_t style, RopeTable t,
                                  void* q, void* k, void* v, int32_t* err, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  const void* a = x;
  if (x_index != nullptr) {  // gather the rows into the workspace first
    const int blocks = (int)(((int64_t)m * 32 + 255) / 256);
    const cudaError_t e = launch_pdl(gather_rows_kernel, blocks, 256, 0, s, (uint8_t*)x_gathered, (const uint8_t*)x,
                                     x_index, m, x_rows, d_model * 2, err);
    if (e != cudaSuccess) return e;
    a = x_gathered;
  }
  ProjParams p;
  p.tokens = tokens;
  p.m = m;
  p.n_tokens = n_tokens;
  p.d_model = d_model;
  p.hq = hq;
  p.hkv = hkv;
  p.head_dim = head_dim;
  p.encode = encode;
  p.style = style;
  p.tab = t.tab;
  p.q = static_cast<uint8_t*>(q);
  p.k = static_cast<uint8_t*>(k);
  p.v = static_cast<uint8_t*>(v);
  p.err = err;
  if (head_dim == 128) return launch_proj_pair<128>(p, a, w, s);
  if (head_dim == 64) return launch_proj_pair<64>(p, a, w, s);
  return cudaErrorInvalidValue;
}

bool qkv_projection_supported(int32_t d_model) { return d_model >= kPK && d_model % kPK == 0; }

cudaError_t launch_projection_timeout_probe(const void* x, int32_t d_model, int32_t m, const void* w, int32_t n_tokens,
                                            int32_t hq, int32_t hkv, void* q, void* k, void* v, int32_t* err,
                                            cudaStream_t s) {
  if (m <= 0 || d_model < 2 * kPK || d_model % kPK != 0) return cudaErrorInvalidValue;  // needs a K step 1
  ProjParams p = {};
  p.m = m;
  p.n_tokens = n_tokens;
  p.d_model = d_model;
  p.hq = hq;
  p.hkv = hkv;
  p.head_dim = 128;
  p.q = static_cast<uint8_t*>(q);
  p.k = static_cast<uint8_t*>(k);
  p.v = static_cast<uint8_t*>(v);
  p.err = err;
  return launch_proj_pair<128, true>(p, x, w, s);
}

}  // namespace cb
