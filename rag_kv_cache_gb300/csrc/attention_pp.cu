// HKVD causal grouped-query attention for large launches on sm_103a: two query tiles per CTA
// whose softmax and tensor-core work alternate ("ping-pong").
//
// What it computes is what attention.cu computes ("数学推导" §形式化, the attention over the
// fused cache; "rag的kvcache问题" §transformer训练与推理并行计算的差异 for the causal mask and
// §阶段二 for computing only the selected rows):
//   out[i, h] = sum_{j <= q_pos[i]} softmax_j(scale * q[i, h] . k[j, g]) v[j, g],  g = h / G.
//
// Tiling. One CTA owns one kv head g and two query tiles of 128 rows each (tile i: TQ = 128 / G
// tokens times the G query heads of g, tokens t0 + i TQ ...), 256 query rows in all, and visits
// the key tiles (128 keys) up to the larger query position of the two. Every K and V tile it
// loads serves both query tiles.
//
// Why two tiles. With one query tile per CTA, the scores of the next key tile can only be
// formed once the softmax of the current one has written P, so the tensor core waits for the
// softmax once per key tile. Here softmax warpgroup i owns query tile i whole (thread r = row r,
// all 128 keys of each key tile) and the issuer alternates between the tiles:
//     P_0(j) ready -> O_0 += P_0(j) V_j, then S_0(j+1) = Q_0 K_{j+1}^T
//     P_1(j) ready -> O_1 += P_1(j) V_j, then S_1(j+1) = Q_1 K_{j+1}^T
// so while warpgroup 0 turns S_0(j+1) into P_0(j+1), the tensor core runs tile 1's products, and
// the other way round: each softmax hides behind the other tile's 16 MMAs, and the two
// warpgroups' exponentials (the MUFU pipe) take turns instead of competing.
//
// Roles (384 threads):
//   WG0, WG1 (warps 0-7)  softmax of query tile 0 / 1 (TMEM lane = row); 224 registers each
//                         (setmaxnreg), since a row's 128 scores are held at once
//   warp 8   initialises the barriers, requests Q_0, Q_1, K_0 and V_0 at entry, then produces
//            the K ring (2 stages; stage j % 2 is refilled once S_1(j) is complete)
//   warp 9   the MMA issuer (one elected lane; tcgen05.mma kind::f16, bf16 in, fp32 accumulate)
//   warp 10  produces the V ring (2 stages; refilled once P_1(j) V_j is complete)
//   warp 11  the issuer's waiter: polls the TMA barriers a round needs and publishes them
// WG2 (warps 8-11) runs with 56 registers (setmaxnreg). Issuer, waiter and WG0 meet on named
// barrier 3 once per key tile (WG0's P_0(j) is in TMEM), issuer and WG1 on named barrier 4.
// TMEM columns: S_0 at 0, S_1 at 128 (fp32, 128 keys); P_i(j) (bf16 pairs, 64 columns) is written
// over the first half of S_i(j) once it has been read; O_0 at 256, O_1 at 256 + D.
// tcgen05.mma operations from one thread run in issue order, so S_i(j+1), issued right after
// P_i(j) V_j, overwrites P_i(j) only after that product has read it.
//
// Barriers are per ring stage (j % 2), so no wait can see a phase two steps ahead of the one it
// wants: S_i(j) completes s_full[i][j % 2] (S_1(j) also frees K stage j % 2), P_i(j) V_j
// completes o_done[i][j % 2] (for i = 1 also frees V stage j % 2).
//
// Every mbarrier wait is bounded (2 s by the global timer); a wait that gives up records a
// timeout in the error word, raises a CTA-wide abort flag, and the CTA drains its copies and
// tensor-core work and frees its TMEM before returning, as in attention.cu.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tmem_ops.cuh"

namespace cb {
namespace {

constexpr int kBM = 128;      // rows per query tile
constexpr int kTiles = 2;     // query tiles per CTA
constexpr int kBN = 128;      // keys per key tile
constexpr int kStages = 2;    // depth of the K and of the V ring
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;
constexpr int kWarpProducerK = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpProducerV = 10;
constexpr int kWarpWaiter = 11;
constexpr int kBarIssue = 2;  // issuer + waiter (64 threads): the first scores
constexpr int kBarTile0 = 3;  // WG0 + issuer + waiter (192 threads), once per key tile
constexpr int kBarTile1 = 4;  // WG1 + issuer (160 threads), once per key tile
constexpr int kBarEpi0 = 5;   // WG0 alone (epilogue)
constexpr int kBarEpi1 = 6;   // WG1 alone (epilogue)
constexpr int kBarExit = 1;   // all 384 threads, before the tensor memory is freed
constexpr int kBarPos = 7;    // all 384 threads, once the query positions are known
constexpr uint32_t kTmemCols = 512;
constexpr int kSoftmaxRegs = 224;  // per thread of WG0 / WG1 after setmaxnreg.inc
constexpr int kOtherRegs = 56;     // per thread of WG2 after setmaxnreg.dec
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kTileSumLimit = 65536.0f;  // a later tile whose P sum exceeds 2^16 moves the reference

__host__ __device__ constexpr uint32_t col_s(int i) { return (uint32_t)(i * kBN); }
__host__ __device__ constexpr uint32_t col_o(int i, int d) { return 256u + (uint32_t)(i * d); }

struct Bars {
  uint64_t q_full;                   // both query tiles
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t s_full[kTiles][kStages];  // S_i(j) complete (commit); [1][s] also: K stage s free
  uint64_t o_done[kTiles][kStages];  // P_i(j) V_j complete (commit); [1][s] also: V stage s free
  uint64_t drain;
};

struct PPParams {
  const int32_t* pos_idx;  // position of query row t: t < pos_k ? pos_idx[t] : pos_base + (t - pos_k)
  int pos_k;
  int pos_base;
  int wait_prior;
  int mq;
  int n_keys;
  int hq;
  int hkv;
  int group;
  int tq;       // query tokens per tile = 128 / group
  int n_pairs;  // CTAs per kv head
  float scale_log2;
  int32_t* err;
};

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// One row's P for a key tile: P = 2^(s * scale - m_ref) for its 128 scores (m_ref = -inf only for
// a row with nothing visible yet, whose scores are then all -inf), packed to bf16 and written to
// TMEM as 32 columns per 64 keys from taddr_p; returns the row sum of P (fp32, +inf if an exponent
// overflowed).
__device__ __forceinline__ float softmax_p(const uint32_t (&sv)[kBN], float m_ref, float scale_log2,
                                           uint32_t taddr_p) {
  const float neg_m = m_ref == -INFINITY ? 0.0f : -m_ref;
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(neg_m, neg_m);
  uint64_t ps2[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) ps2[q] = f2_pack(0.0f, 0.0f);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int c = 64 * h + 2 * e;
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nm2), x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      ps2[e & 3] = f2_add(ps2[e & 3], f2_pack(p0, p1));
      pk[e] = pack2(p0, p1);
    }
    tmem_st_x32(taddr_p + 32 * h, pk);
  }
  float sa, sb;
  f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), sa, sb);
  return sa + sb;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    hkvd_attention_pp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                             const PPParams p) {
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kQBytes = kBM * D * 2;  // one query tile
  constexpr uint32_t kKVBytes = kBN * D * 2;
  constexpr uint32_t kQBox = kBM * 128;   // bytes of one 64-column box of a query tile
  constexpr uint32_t kKVBox = kBN * 128;  // bytes of one 64-column box of a K or V tile

  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_maxpos;
  __shared__ int s_first_ok;
  __shared__ int s_round_ok[2];

  pdl_launch_dependents();
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;                        // query tile i at sQ + i kQBytes
  const uint32_t sK0 = base + kTiles * kQBytes;    // K stage s at sK0 + s kKVBytes
  const uint32_t sV0 = sK0 + kStages * kKVBytes;   // V stage s at sV0 + s kKVBytes

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int lin = blockIdx.x;
  const int pair = p.n_pairs - 1 - lin / p.hkv;  // later (longer) query tiles first
  const int g = lin % p.hkv;
  const int t0 = pair * kTiles * p.tq;  // first token of tile 0; tile i starts at t0 + i tq
  const bool tile1_rows = t0 + p.tq < p.mq;  // the last pair of an odd tile count has no tile 1

  if (warp == kWarpProducerK && lane == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      for (int i = 0; i < kTiles; ++i) {
        mbar_init(smem_u32(&bars.s_full[i][s]), 1);
        mbar_init(smem_u32(&bars.o_done[i][s]), 1);
      }
    }
    mbar_init(smem_u32(&bars.drain), 1);
    s_abort = 0;
    s_maxpos = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (p.wait_prior) pdl_wait();  // the query rows and fused K/V come from the kernels before
    const uint32_t qb = smem_u32(&bars.q_full);
    mbar_expect_tx(qb, kTiles * kQBytes);
#pragma unroll
    for (int i = 0; i < kTiles; ++i)
#pragma unroll
      for (int b = 0; b < kBoxes; ++b)  // an empty tile 1 reads the fill value past mq
        tma_load_4d(sQ + i * kQBytes + b * kQBox, &tm_q, qb, b * 64, 0, g, t0 + i * p.tq);
    const uint32_t kb = smem_u32(&bars.k_full[0]);
    mbar_expect_tx(kb, kKVBytes);
#pragma unroll
    for (int b = 0; b < kBoxes; ++b) tma_load_3d(sK0 + b * kKVBox, &tm_k, kb, b * 64, g, 0);
    const uint32_t vb = smem_u32(&bars.v_full[0]);
    mbar_expect_tx(vb, kKVBytes);
#pragma unroll
    for (int b = 0; b < kBoxes; ++b) tma_load_3d(sV0 + b * kKVBox, &tm_v, vb, b * 64, g, 0);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;

  if (warp >= kTiles * (kSoftmaxThreads / 32)) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    named_sync(kBarPos, kThreads);  // the softmax warps have read the query positions
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int n_kv = s_maxpos / kBN + 1;  // key tiles the CTA visits
    if (warp == kWarpProducerK && lane == 0) {
      const uint32_t qb = smem_u32(&bars.q_full);
      int nk = 1;  // K tile 0 is in flight already
      for (int j = 1; j < n_kv; ++j) {
        const int st = j % kStages;
        // K_{j-2} held this stage: free once S_1(j-2) (issued after S_0(j-2)) is complete
        if (j >= kStages &&
            !mbar_wait_inl(smem_u32(&bars.s_full[1][st]), ((j / kStages) - 1) & 1, abort_flag, p.err, 1))
          break;
        const uint32_t kb = smem_u32(&bars.k_full[st]);
        mbar_expect_tx(kb, kKVBytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b)
          tma_load_3d(sK0 + st * kKVBytes + b * kKVBox, &tm_k, kb, b * 64, g, j * kBN);
        nk = j + 1;
      }
      // Before the CTA can exit, every copy issued must have landed.
      mbar_wait_inl(qb, 0, abort_flag, p.err, 3, false);
      for (int j = nk - kStages < 0 ? 0 : nk - kStages; j < nk; ++j)
        mbar_wait_inl(smem_u32(&bars.k_full[j % kStages]), (j / kStages) & 1, abort_flag, p.err, 4, false);
    } else if (warp == kWarpProducerV && lane == 0) {
      int nv = 1;  // V tile 0 is in flight already
      for (int j = 1; j < n_kv; ++j) {
        const int st = j % kStages;
        // V_{j-2} held this stage: free once P_1(j-2) V_{j-2} (after P_0(j-2) V_{j-2}) is complete
        if (j >= kStages &&
            !mbar_wait_inl(smem_u32(&bars.o_done[1][st]), ((j / kStages) - 1) & 1, abort_flag, p.err, 2))
          break;
        const uint32_t vb = smem_u32(&bars.v_full[st]);
        mbar_expect_tx(vb, kKVBytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b)
          tma_load_3d(sV0 + st * kKVBytes + b * kKVBox, &tm_v, vb, b * 64, g, j * kBN);
        nv = j + 1;
      }
      for (int j = nv - kStages < 0 ? 0 : nv - kStages; j < nv; ++j)
        mbar_wait_inl(smem_u32(&bars.v_full[j % kStages]), (j / kStages) & 1, abort_flag, p.err, 5, false);
    } else if (warp == kWarpWaiter) {
      // The TMA inputs of the first scores (Q_0, Q_1, K_0), then per key tile j those of round j
      // (V_j and K_{j+1}), published to the issuer through shared memory before it meets the
      // issuer (and WG0) on a named barrier. Every round is joined, also after a failure.
      auto spin_all = [&](uint32_t bar, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, mbar_spin_inl(bar, parity, abort_flag, p.err, site));
      };
      bool ok = spin_all(smem_u32(&bars.q_full), 0, 10) && spin_all(smem_u32(&bars.k_full[0]), 0, 11);
      if (lane == 0) s_first_ok = ok ? 1 : 0;
      __syncwarp();  // bar.sync is warp-aligned: reach it converged
      named_sync(kBarIssue, 64);
      for (int j = 0; j < n_kv; ++j) {
        ok = ok && spin_all(smem_u32(&bars.v_full[j % kStages]), (j / kStages) & 1, 13) &&
             (j + 1 >= n_kv || spin_all(smem_u32(&bars.k_full[(j + 1) % kStages]), ((j + 1) / kStages) & 1, 12));
        if (lane == 0) s_round_ok[j & 1] = ok ? 1 : 0;
        __syncwarp();
        named_sync(kBarTile0, 192);
      }
    } else if (warp == kWarpMma) {
      constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false);
      constexpr uint32_t idesc_o = idesc_bf16(kBM, D, true);
      const uint64_t dk0 = sdesc(sK0, 16, 1024);
      const uint64_t dv0 = sdesc(sV0, kKVBox, 1024);
      // S_i(j) = Q_i K_j^T into S_i; elected lane only.
      auto issue_s = [&](int i, int j) {
        const int st = j % kStages;
        const uint64_t dq = sdesc(sQ + i * kQBytes, 16, 1024);
        const uint64_t dk = dk0 + (uint64_t)((st * kKVBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int bx = ks / 4, kk = ks % 4;
          mma_ss(tmem + col_s(i), dq + (uint64_t)((bx * kQBox + kk * 32) >> 4),
                 dk + (uint64_t)((bx * kKVBox + kk * 32) >> 4), idesc_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&bars.s_full[i][st]));
      };
      // O_i (+)= P_i(j) V_j: P from TMEM (16 keys = 8 columns per MMA), V MN-major in shared memory.
      auto issue_pv = [&](int i, int j) {
        const int st = j % kStages;
        const uint64_t dv = dv0 + (uint64_t)((st * kKVBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          mma_ts(tmem + col_o(i, D), tmem + col_s(i) + ks * 8, dv + (uint64_t)((ks * 16 * 128) >> 4), idesc_o,
                 (ks > 0 || j > 0) ? 1u : 0u);
        tc_commit(smem_u32(&bars.o_done[i][st]));
      };
      __syncwarp();
      named_sync(kBarIssue, 64);
      bool ok = s_first_ok != 0;
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          issue_s(0, 0);
          issue_s(1, 0);
        }
        __syncwarp();
      }
      for (int j = 0; j < n_kv; ++j) {
        __syncwarp();
        named_sync(kBarTile0, 192);  // P_0(j) in TMEM; V_j and K_{j+1} loaded (waiter)
        ok = ok && s_round_ok[j & 1] != 0 && !*abort_flag;
        if (ok) {
          tc_fence_after();
          if (elect_one()) {
            issue_pv(0, j);
            if (j + 1 < n_kv) issue_s(0, j + 1);
          }
          __syncwarp();
        }
        __syncwarp();
        named_sync(kBarTile1, 160);  // P_1(j) in TMEM
        ok = ok && !*abort_flag;
        if (ok) {
          tc_fence_after();
          if (elect_one()) {
            issue_pv(1, j);
            if (j + 1 < n_kv) issue_s(1, j + 1);
          }
          __syncwarp();
        }
      }
      // All tensor-core work issued by this CTA completes before TMEM is freed.
      if (elect_one()) tc_commit(smem_u32(&bars.drain));
      __syncwarp();
      mbar_wait_inl(smem_u32(&bars.drain), 0, abort_flag, p.err, 14, false);
    }
    // The two register regions end separately (no common tail after the branch): every warp
    // meets on named barrier 1 before warp 0 frees the tensor memory.
    __syncwarp();
    tc_fence_before();
    named_sync(kBarExit, kThreads);
    return;
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    if (p.wait_prior) pdl_wait();  // the positions come from the kernels before this one
    // Query position of each softmax thread's row; rows past the tile's last token repeat it (an
    // empty tile 1 repeats token mq - 1); those rows are never stored.
    int my_pos = 0;
    {
      const int ti = threadIdx.x / kSoftmaxThreads, r = threadIdx.x % kSoftmaxThreads;
      const int tfirst = t0 + ti * p.tq;
      const int t_last = min(tfirst + p.tq, p.mq) - 1;
      const int t = min(tfirst + r / p.group, t_last);
      auto qpos = [&](int tt) { return tt < p.pos_k ? p.pos_idx[tt] : p.pos_base + (tt - p.pos_k); };
      int pos = qpos(t);
      if (pos < 0 || pos >= p.n_keys) {
        if (r % p.group == 0) record_error(p.err, kErrIndex, t);
        pos = pos < 0 ? 0 : p.n_keys - 1;
      }
      if (r % p.group == 0 && t == tfirst + r / p.group && t > 0 && qpos(t - 1) >= pos)
        record_error(p.err, kErrOrder, t);
      atomicMax(&s_maxpos, pos);
      my_pos = pos;
    }
    tc_fence_before();
    named_sync(kBarPos, kThreads);
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int n_kv = s_maxpos / kBN + 1;  // key tiles the CTA visits
    const int ti = warp / 4;  // this warpgroup's query tile
    const int r = threadIdx.x % kBM;
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    float m_ref = -INFINITY, l = 0.0f;  // reference max (log2 units) that O_ti and l are scaled to
    bool ok = true;
    auto wait_o = [&](int j, int site) -> bool {
      const bool w = mbar_spin_inl(smem_u32(&bars.o_done[ti][j % kStages]), (j / kStages) & 1, abort_flag, p.err, site);
      return __all_sync(0xffffffffu, w);
    };
    // One key tile; false if a wait gave up (the abort flag is raised then).
    auto tile = [&](int j) -> bool {
      if (!__all_sync(0xffffffffu, mbar_spin_inl(smem_u32(&bars.s_full[ti][j % kStages]), (j / kStages) & 1,
                                             abort_flag, p.err, 20 + ti)))
        return false;
      tc_fence_after();
      uint32_t sv[kBN];  // this row's 128 scores
      {
        uint32_t(&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t(&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        uint32_t(&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[64]);
        uint32_t(&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[96]);
        tmem_ld_x32_async(lane_base + col_s(ti), s0);
        tmem_ld_x32_async(lane_base + col_s(ti) + 32, s1);
        tmem_ld_x32_async(lane_base + col_s(ti) + 64, s2);
        tmem_ld_x32_async(lane_base + col_s(ti) + 96, s3);
        tmem_wait_ld(s0);
        tmem_wait_ld(s1);
        tmem_wait_ld(s2);
        tmem_wait_ld(s3);
      }
      const int lim = my_pos - j * kBN;  // columns c <= lim are visible to this row
      if (__any_sync(0xffffffffu, lim < kBN - 1)) {  // diagonal tiles only
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > lim) sv[c] = 0xff800000u;  // -inf
      }
      // P = 2^(s * scale - m_ref), packed to bf16 and written over the first half of S_ti (32
      // columns per 64 keys), and its row sum. A row's first visible tile sets the reference m_ref
      // to the tile's max. Later tiles run the exponentials against the reference without taking
      // their max first (the softmax sets the round's pace): a tile whose row sum stays within
      // 2^16 has every P within 2^16, far from overflow in P, O and l. A tile whose sum passes
      // that (its max grew by more than 2^9) takes its max, moves the reference of the rows whose
      // max passes it by more than 2^8, rescales O and computes P again before the issuer reads it.
      const uint32_t taddr_p = lane_base + col_s(ti);
      bool move_ref = !__all_sync(0xffffffffu, m_ref != -INFINITY);  // a row's first visible tile
      float sum = 0.0f;
      if (!move_ref) {
        sum = softmax_p(sv, m_ref, p.scale_log2, taddr_p);
        move_ref = !__all_sync(0xffffffffu, sum <= kTileSumLimit);  // rare: the max jumped
      }
      if (move_ref) {
        // Four independent chains of three-input max.
        float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kBN; c += 8) {
          tm[0] = max3(tm[0], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
          tm[1] = max3(tm[1], __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
          tm[2] = max3(tm[2], __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
          tm[3] = max3(tm[3], __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
        }
        const float mt = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])) * p.scale_log2;  // -inf: nothing visible
        const bool up = mt > m_ref + kRescaleThreshold;  // always, at a row's first visible key
        if (__any_sync(0xffffffffu, up)) {
          const float alpha = up ? ex2(m_ref - mt) : 1.0f;  // 0 for a row that had nothing visible
          const bool scale_o = up && m_ref != -INFINITY;
          if (up) {
            l *= alpha;
            m_ref = mt;
          }
          // O_ti holds the sum through tile j - 1: wait for that product, then scale it.
          if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
            if (!wait_o(j - 1, 22 + ti)) return false;
            tc_fence_after();
            const float a = scale_o ? alpha : 1.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld_x32(lane_base + col_o(ti, D) + c0, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
              tmem_st_x32(lane_base + col_o(ti, D) + c0, o);
            }
            tmem_st_wait();
          }
        }
        sum = softmax_p(sv, m_ref, p.scale_log2, taddr_p);  // these stores replace any earlier P
      }
      l += sum;
      tmem_st_wait();
      return true;
    };
    // Every softmax warp syncs once per key tile on its tile's named barrier, also after a failed
    // wait (then without work), so every round of the issuer and the waiter completes.
    for (int j = 0; j < n_kv; ++j) {
      if (ok) ok = tile(j);
      tc_fence_before();
      __syncwarp();
      if (ti == 0)
        named_sync(kBarTile0, 192);
      else
        named_sync(kBarTile1, 160);
    }
    if (ok) ok = wait_o(n_kv - 1, 26 + ti);
    ok = ok && !*abort_flag;
    // Epilogue: out = O_ti / l, staged in this tile's Q buffer (every product that reads Q is
    // complete once the last P_ti V has completed) as the output box's 128-byte swizzled rows.
    constexpr uint32_t kOutBox = kBM * 128;
    const uint32_t sOut = sQ + ti * kQBytes;
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv = 1.0f / l;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 64) {
        uint32_t o0[32], o1[32];
        tmem_ld_x32_async(lane_base + col_o(ti, D) + c0, o0);
        tmem_ld_x32_async(lane_base + col_o(ti, D) + c0 + 32, o1);
        tmem_wait_ld(o0);
        tmem_wait_ld(o1);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(q < 4 ? o0[q * 8 + e] : o1[(q - 4) * 8 + e]) * inv;
          const uint4 pk = pack8(f);
          const int c = c0 + q * 8;
          const uint32_t dst = sOut + (uint32_t)(c / 64) * kOutBox + (uint32_t)r * 128u +
                               (uint32_t)((((c % 64) / 8) ^ (r & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk.x), "r"(pk.y), "r"(pk.z),
                       "r"(pk.w)
                       : "memory");
        }
      }
    }
    // The tile's rows are one box of the output per 64 columns (TQ tokens x G heads); rows past
    // mq are clipped by the tensor map, and an empty tile 1 stores nothing.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (ti == 0)
      named_sync(kBarEpi0, kSoftmaxThreads);
    else
      named_sync(kBarEpi1, kSoftmaxThreads);
    if (r == 0 && !*abort_flag && (ti == 0 || tile1_rows)) {
#pragma unroll
      for (int b = 0; b < kBoxes; ++b)
        asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                         &tm_o),
                     "r"(b * 64), "r"(0), "r"(g), "r"(t0 + ti * p.tq), "r"(sOut + b * kOutBox)
                     : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the box has left shared memory
    }
    __syncwarp();
    tc_fence_before();
    named_sync(kBarExit, kThreads);
    if (warp == 0) {
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
  }
}

}  // namespace

bool attention_pp_eligible(int32_t mq, int32_t hq, int32_t hkv, int32_t head_dim) {
  if (head_dim != 128 || hq % hkv != 0 || mq <= 0) return false;
  const int group = hq / hkv;
  if (kBM % group != 0) return false;
  const int tq = kBM / group;
  const int64_t n_qtiles = ((int64_t)mq + tq - 1) / tq;
  const int64_t ctas = (n_qtiles + kTiles - 1) / kTiles * hkv;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
    else
      return false;
  }
  // At least 1.5 waves of its 256-row CTAs. Measured crossovers: at 1.79 waves (the Llama-70B shape's
  // later layers) the paired kernel runs the layer in 126.5 against 132.8 us; at 1.11 (the ratio
  // sweep at 15%) it loses, 111.1 against 82.4 us, since one tile per CTA then fills more SMs.
  return 2 * ctas >= 3 * (int64_t)sms;
}

cudaError_t launch_hkvd_attention_pp(const void* q, QueryPositions qp, int32_t mq, const void* k, const void* v,
                                     int32_t n_keys, int32_t hq, int32_t hkv, float scale, void* out, int32_t* err,
                                     cudaStream_t s) {
  constexpr int D = 128;
  if (mq <= 0) return cudaSuccess;
  const int group = hq / hkv;
  const int tq = kBM / group;
  const int n_qtiles = (mq + tq - 1) / tq;
  const int n_pairs = (n_qtiles + kTiles - 1) / kTiles;
  // The register split: the block is launched with numRegs per thread and setmaxnreg moves them
  // between the warpgroups; a kernel built with fewer registers than the split needs would wait
  // forever in setmaxnreg.inc, so it is never launched (the caller then uses the other kernel).
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, hkvd_attention_pp_kernel<D>);
    if (e != cudaSuccess) return e;
    regs = a.numRegs;
  }
  if (regs * kThreads < kTiles * kSoftmaxThreads * kSoftmaxRegs + kSoftmaxThreads * kOtherRegs)
    return cudaErrorNotSupported;
  CUtensorMap tq_map, tk_map, tv_map, to_map;
  const cuuint64_t qd[4] = {(cuuint64_t)D, (cuuint64_t)group, (cuuint64_t)hkv, (cuuint64_t)mq};
  const cuuint64_t qs[3] = {(cuuint64_t)D * 2, (cuuint64_t)group * D * 2, (cuuint64_t)hq * D * 2};
  const cuuint32_t qb[4] = {64, (cuuint32_t)group, 1, (cuuint32_t)tq};
  const cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)n_keys};
  const cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
  const cuuint32_t kbx[3] = {64, 1, (cuuint32_t)kBN};
  if (!encode_map(&tq_map, q, 4, qd, qs, qb) || !encode_map(&tk_map, k, 3, kd, ks, kbx) ||
      !encode_map(&tv_map, v, 3, kd, ks, kbx) || !encode_map(&to_map, out, 4, qd, qs, qb))
    return cudaErrorInvalidValue;
  PPParams p;
  p.pos_idx = qp.idx;
  p.pos_k = qp.k;
  p.pos_base = qp.base;
  p.wait_prior = qp.wait_prior ? 1 : 0;
  p.mq = mq;
  p.n_keys = n_keys;
  p.hq = hq;
  p.hkv = hkv;
  p.group = group;
  p.tq = tq;
  p.n_pairs = n_pairs;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = err;
  const size_t smem = 1024 + (size_t)(kTiles * kBM + 2 * kStages * kBN) * D * 2;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = set_smem_limit_once(hkvd_attention_pp_kernel<D>, (int)smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(hkvd_attention_pp_kernel<D>, n_pairs * hkv, kThreads, smem, s, tq_map, tk_map, tv_map, to_map,
                    p);
}

}  // namespace cb
