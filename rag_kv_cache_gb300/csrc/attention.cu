// HKVD causal grouped-query attention on sm_103a: TMA loads, tcgen05.mma with
// TMEM accumulators, online softmax with one thread per query row.
//
// What it computes ("数学推导" §形式化, the attention over the fused cache;
// "rag的kvcache问题" §transformer训练与推理并行计算的差异 for the causal mask and
// §阶段二 for computing only the selected rows):
//   out[i, h] = sum_{j <= q_pos[i]} softmax_j(scale * q[i, h] . k[j, g]) v[j, g],  g = h / G.
//
// Tiling. One CTA owns one kv head g and 128 query rows: TQ = 128 / G query
// tokens times the G query heads that share g (row r = token r / G, head r % G),
// so every K/V tile it loads serves all G heads. Key tiles are 128 keys; the
// CTA visits key tiles 0 .. (largest query position in the tile) / 128.
//
// Roles (384 threads):
//   WG0, WG1 (warps 0-7) softmax: thread r of each owns query row r (TMEM lane
//              r); WG h takes keys [64h, 64h + 64) of every key tile, with its
//              own running max / sum and its own O accumulator, so the two
//              halves of a tile are exponentiated at the same time; the two
//              partial results are merged in the epilogue.
//   warp 8     initialises the barriers and requests Q, K_0 and V_0 at entry, then
//              is the TMA producer of the K tiles (3-stage ring; a stage is
//              refilled as soon as its S = Q K^T is done);
//   warp 9     issuer of both products (tcgen05.mma, bf16 in, fp32 accumulate);
//   warp 10    TMA producer of V tiles (3-stage ring, refilled after P V);
//   warp 11    the issuer's waiter: it polls the TMA barriers a round of MMAs
//              depends on; the issuer, the waiter and the softmax warps meet on a
//              named barrier per tile (the softmax warps once their P is in TMEM).
//              A warp that has just issued MMAs waits
//              100-200 cycles on its next shared-memory access (an mbarrier test
//              included) while a named barrier returns at once, so the issuer
//              itself never touches an mbarrier in the tile loop.
// TMEM columns: S in two buffers, tile j in buffer j % 2 at 128 (j % 2) (one
// N = 128 MMA chain per key tile; WG h reads its 64 columns); each warpgroup
// writes its P_j (bf16 pairs, 32 columns) over the first half of its own S_j
// columns once it has copied them out; O accumulators at 256 and 256 + D.
// One thread issues every MMA, and tcgen05.mma operations from one thread run
// in issue order: S_{j+2} is issued into buffer j % 2 right after P V_j, which
// reads P_j from it, with no completion wait in between, so the tensor core
// always has the next scores queued behind the current P V while the softmax
// works on tile j + 1. The softmax never hands a buffer back: S_j is consumed
// before P_j is written, and P_j before S_{j+2} overwrites it, by construction.
// The issuing warp runs converged and one elected lane issues, so the loop
// index, stages and operand descriptors are warp-uniform values in uniform
// registers; descriptors are formed once and advanced by compile-time offsets.
//
// Every mbarrier wait is bounded (2 s by the global timer). A wait that gives
// up records a timeout in the error word, raises a CTA-wide abort flag that
// ends the other roles' loops, and the CTA drains its tensor-core work and
// frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "attn_common.cuh"
#include "tc_common.cuh"
#include "tmem_ops.cuh"

namespace cb {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;     // keys per tile
constexpr int kHalf = kBN / 2;  // keys of a tile per softmax warpgroup
constexpr int kKStages = 3;  // depth of the K ring
constexpr int kVStages = 3;  // depth of the V ring (Q + 3 K + 3 V tiles = 224 KiB for D = 128): a V
                             // stage is refilled only after its P V completes, so a load has two
                             // tiles of lead before its P V
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;  // per softmax warpgroup
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpProducerV = 10;
constexpr int kWarpWaiter = 11;
constexpr int kBarIssue = 2;  // named barrier: issuer + waiter (64 threads), the first round
constexpr int kBarRound = 3;  // named barrier: the softmax warps + issuer + waiter, once per tile
constexpr int kRoundThreads = 2 * 128 + 64;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S (fp32) buffer b at 128 b, warpgroup h's half at +64 h (P_j over the first 32
// columns of that half); O accumulators at 256 + h D.
__host__ __device__ constexpr uint32_t col_s(int b, int h) { return (uint32_t)(b * kBN + h * kHalf); }
__host__ __device__ constexpr uint32_t col_o(int h, int d) { return 256u + (uint32_t)(h * d); }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kTileSumLimit = 65536.0f;  // a later tile whose P sum exceeds 2^16 moves the reference

// One MMA commit per product: S_j's completion frees K stage j % 3 and tells the softmax that S_j
// is in TMEM (both wait on s_done[j % 3], phase j / 3); P V_j's completion frees V stage j % 3 and
// tells the softmax that O holds tile j (pv_done[j % 3]). A commit costs the tensor pipe ~30
// cycles, so sharing one barrier between the two waiters of each product saves two per round.
// The phases cannot alias: S_{j+3} is issued only after the softmax has finished tile j + 1, and
// P V_{j+3} only after it has finished tile j + 3.
static_assert(kKStages == 3 && kVStages == 3, "the S and P V barriers are indexed by the K and V stages");
struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKStages];
  uint64_t s_done[kKStages];  // S_j complete: K stage j % 3 free and S_j readable (MMA commit)
  uint64_t v_full[kVStages];
  uint64_t pv_done[kVStages];  // P V_j complete: V stage j % 3 free and O updated (MMA commit)
  uint64_t drain;
};

struct Params {
  // Position of query row t: t < pos_k ? pos_idx[t] : pos_base + (t - pos_k).
  const int32_t* pos_idx;
  int pos_k;
  int pos_base;
  int wait_prior;  // 1: wait for the previous kernel on the stream before reading (programmatic launch)
  int mq;
  int n_keys;
  int hq;
  int hkv;
  int group;     // query heads per kv head
  int tq;        // query tokens per tile = 128 / group
  int n_qtiles;
  float scale_log2;
  uint8_t* out;
  int32_t* err;
  // Diagnostics (null in the blend): row_stats receives each row's (reference, sum) of the softmax
  // in log2 units, A_ij = 2^(s_ij * scale_log2 - reference) / sum (the reference is the softmax's
  // own, at most 16 below the row's max). The counting instance reads count_stats
  // (such a pair per row) and writes to counts, per row, how many of the n_keys weights lie
  // below 2^log2_eps (masked keys, weight 0, included).
  float2* row_stats;
  const float2* count_stats;
  float log2_eps;
  int32_t* counts;
};

// PROBE: the wait-timeout probe (test support only): the K producer never requests key tile 1
// and every wait gives up after kProbeTimeoutNs, so the CTA takes its failure path (timeout
// recorded, remaining rounds skipped, copies and tensor-core work drained, TMEM freed).
// One row's P for its half of a key tile: P = 2^(s * scale - m_ref) for its 64 scores (m_ref = -inf
// only for a row with nothing visible yet, whose scores are then all -inf), packed to bf16 into pk
// (key 2e in the low half of pk[e]); returns the row sum of P (fp32, +inf if an exponent overflowed).
__device__ __forceinline__ float softmax_p(const uint32_t (&sv)[kHalf], float m_ref, float scale_log2,
                                           uint32_t (&pk)[kHalf / 2]) {
  const float neg_m = m_ref == -INFINITY ? 0.0f : -m_ref;
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(neg_m, neg_m);
  uint64_t ps2[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) ps2[q] = f2_pack(0.0f, 0.0f);
#pragma unroll
  for (int e = 0; e < kHalf / 2; ++e) {
    float t0, t1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sc2, nm2), t0, t1);
    const float p0 = ex2(t0), p1 = ex2(t1);
    ps2[e & 3] = f2_add(ps2[e & 3], f2_pack(p0, p1));
    pk[e] = pack2(p0, p1);
  }
  float sa, sb;
  f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), sa, sb);
  return sa + sb;
}

template <int D, bool COUNT, bool PROBE = false>
__global__ void __maxnreg__(128)
    hkvd_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                          const Params p) {
  constexpr int kBoxes = D / 64;
  constexpr uint32_t kQBytes = kBM * D * 2;
  constexpr uint32_t kKVBytes = kBN * D * 2;
  constexpr uint32_t kQBox = kBM * 128;   // bytes of one 64-column box of Q
  constexpr uint32_t kKVBox = kBN * 128;  // bytes of one 64-column box of a K or V tile
  constexpr uint64_t kLimit = PROBE ? kProbeTimeoutNs : kTimeoutNs;

  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_maxpos;
  // waiter -> issuer: the TMA inputs of the first round / of round j (slot j % 2) are in shared
  // memory (0: a wait gave up). Two slots: the waiter's write for round j + 1 cannot overtake the
  // issuer's read for round j, which precedes its arrival for round j + 1.
  __shared__ int s_first_ok;   // Q and K_0 are in (S_0 may be issued)
  __shared__ int s_second_ok;  // K_1 is in too (S_1 may be issued)
  __shared__ int s_round_ok[2];

  pdl_launch_dependents();
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK0 = base + kQBytes;
  const uint32_t sV0 = sK0 + kKStages * kKVBytes;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int lin = blockIdx.x;
  const int tile = p.n_qtiles - 1 - lin / p.hkv;  // later (longer) query tiles first
  const int g = lin % p.hkv;
  const int t0 = tile * p.tq;
  const int t_last = min(t0 + p.tq, p.mq) - 1;

  // The producer thread initialises the barriers and starts the loads of Q and of the first K and
  // V tiles at once: they do not depend on the query positions (every query tile sees key tile 0),
  // so they overlap warp 0's TMEM allocation and the softmax threads' reads of the positions.
  if (warp == kWarpProducer && lane == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.s_done[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.pv_done[s]), 1);
    }
    mbar_init(smem_u32(&bars.drain), 1);
    s_abort = 0;
    s_maxpos = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // The query rows and fused K/V come from the kernels before this one on the stream.
    if (p.wait_prior) pdl_wait();
    const uint32_t qb = smem_u32(&bars.q_full);
    mbar_expect_tx(qb, kQBytes);
#pragma unroll
    for (int b = 0; b < kBoxes; ++b) tma_load_4d(sQ + b * kQBox, &tm_q, qb, b * 64, 0, g, t0);
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
  // The positions come from the kernels before this one on the stream.
  if (p.wait_prior) pdl_wait();

  // Query position of each softmax thread's row; padded rows repeat the tile's last token.
  int my_pos = 0;
  if (threadIdx.x < 2 * kSoftmaxThreads) {
    const int r = threadIdx.x % kBM;
    const int t = min(t0 + r / p.group, t_last);
    auto qpos = [&](int tt) { return tt < p.pos_k ? p.pos_idx[tt] : p.pos_base + (tt - p.pos_k); };
    int pos = qpos(t);
    if (pos < 0 || pos >= p.n_keys) {
      if (threadIdx.x < kSoftmaxThreads) record_error(p.err, kErrIndex, t);
      pos = pos < 0 ? 0 : p.n_keys - 1;
    }
    if (threadIdx.x < kSoftmaxThreads) {
      if (r % p.group == 0 && t == t0 + r / p.group && t > 0 && qpos(t - 1) >= pos)
        record_error(p.err, kErrOrder, t);
      atomicMax(&s_maxpos, pos);
    }
    my_pos = pos;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int n_kv = s_maxpos / kBN + 1;  // key tiles the query tile sees
  volatile int* abort_flag = &s_abort;

  if (warp >= 2 * (kSoftmaxThreads / 32)) {
    if (warp == kWarpProducer && lane == 0) {
      const uint32_t qb = smem_u32(&bars.q_full);
      int nk = 1;  // Q and K tile 0 are in flight already
      for (int j = 1; j < n_kv; ++j) {
        const int sk = j % kKStages;
        if (j >= kKStages &&
            !mbar_wait(smem_u32(&bars.s_done[sk]), ((j / kKStages) - 1) & 1, abort_flag, p.err, 1, true, kLimit))
          break;
        if constexpr (PROBE) {
          if (j == 1) {  // never requested: every wait on this tile runs into its limit
            nk = j + 1;
            continue;
          }
        }
        const uint32_t kb = smem_u32(&bars.k_full[sk]);
        mbar_expect_tx(kb, kKVBytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b)
          tma_load_3d(sK0 + sk * kKVBytes + b * kKVBox, &tm_k, kb, b * 64, g, j * kBN);
        nk = j + 1;
      }
      // Before the CTA can exit, every copy issued must have landed.
      mbar_wait(qb, 0, abort_flag, p.err, 3, false, kLimit);
      for (int j = nk - kKStages < 0 ? 0 : nk - kKStages; j < nk; ++j)
        mbar_wait(smem_u32(&bars.k_full[j % kKStages]), (j / kKStages) & 1, abort_flag, p.err, 4, false, kLimit);
    } else if (warp == kWarpProducerV && lane == 0) {
      int nv = 1;  // V tile 0 is in flight already
      for (int j = 1; j < n_kv; ++j) {
        const int sv = j % kVStages;
        if (j >= kVStages &&
            !mbar_wait(smem_u32(&bars.pv_done[sv]), ((j / kVStages) - 1) & 1, abort_flag, p.err, 2, true, kLimit))
          break;
        const uint32_t vb = smem_u32(&bars.v_full[sv]);
        mbar_expect_tx(vb, kKVBytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b)
          tma_load_3d(sV0 + sv * kKVBytes + b * kKVBox, &tm_v, vb, b * 64, g, j * kBN);
        nv = j + 1;
      }
      for (int j = nv - kVStages < 0 ? 0 : nv - kVStages; j < nv; ++j)
        mbar_wait(smem_u32(&bars.v_full[j % kVStages]), (j / kVStages) & 1, abort_flag, p.err, 5, false, kLimit);
    } else if (warp == kWarpMma || warp == kWarpWaiter) {
      // Rounds: round -1 issues S_0 (once Q and K_0 are in) and then S_1 (once K_1 is, after a
      // second meeting of issuer and waiter); round j issues P V_j and then S_{j+2} into the same
      // buffer. The waiter polls the TMA barriers a round needs (Q and K_0, K_1; then V_j and
      // K_{j+2}) and publishes whether they completed; the issuer and the waiter then meet the
      // softmax warps, whose joining says P_j is in TMEM, on named barrier kBarRound (round -1:
      // kBarIssue, issuer and waiter only). A named barrier completes within cycles of its last
      // arrival; an mbarrier polled by a busy warp was noticed hundreds of cycles late.
      if (warp == kWarpWaiter) {
        auto spin_all = [&](uint32_t bar, uint32_t parity, int site) -> bool {
          return __all_sync(0xffffffffu, mbar_spin(bar, parity, abort_flag, p.err, site, kLimit));
        };
        auto k_ready = [&](int j) {
          return spin_all(smem_u32(&bars.k_full[j % kKStages]), (j / kKStages) & 1, 11);
        };
        // S_0 goes out as soon as Q and K_0 are in, S_1 once K_1 is (it was requested after the
        // query positions were known).
        bool ok = spin_all(smem_u32(&bars.q_full), 0, 10) && k_ready(0);
        if (lane == 0) s_first_ok = ok ? 1 : 0;
        // bar.sync is warp-aligned: the warp must reach it converged, not split by the lane-0
        // store above (a split warp's arrivals can be counted in the wrong phase).
        __syncwarp();
        asm volatile("bar.sync %0, 64;" ::"n"(kBarIssue) : "memory");
        if (n_kv > 1) {
          ok = ok && k_ready(1);
          if (lane == 0) s_second_ok = ok ? 1 : 0;
          __syncwarp();
          asm volatile("bar.sync %0, 64;" ::"n"(kBarIssue) : "memory");
        }
        for (int j = 0; j < n_kv; ++j) {
          // every round is joined, also after a failure (the issuer then skips its MMAs)
          ok = ok && spin_all(smem_u32(&bars.v_full[j % kVStages]), (j / kVStages) & 1, 13) &&
               (j + 2 >= n_kv || k_ready(j + 2));
          if (lane == 0) s_round_ok[j & 1] = ok ? 1 : 0;
          __syncwarp();
          asm volatile("bar.sync %0, %1;" ::"n"(kBarRound), "n"(kRoundThreads) : "memory");
        }
      } else {
        constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false);
        constexpr uint32_t idesc_o = idesc_bf16(kBM, D, true);
        const uint64_t dq = sdesc(sQ, 16, 1024);
        const uint64_t dk0 = sdesc(sK0, 16, 1024);
        const uint64_t dv0 = sdesc(sV0, kKVBox, 1024);
        // S_j = Q K_j^T into buffer j % 2; elected lane only.
        auto issue_s = [&](int j) {
          const int st = j % kKStages, b = j & 1;
          const uint64_t dk = dk0 + (uint64_t)((st * kKVBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int bx = ks / 4, kk = ks % 4;
            mma_ss(tmem + col_s(b, 0), dq + (uint64_t)((bx * kQBox + kk * 32) >> 4),
                   dk + (uint64_t)((bx * kKVBox + kk * 32) >> 4), idesc_s, ks > 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&bars.s_done[st]));
        };
        __syncwarp();
        asm volatile("bar.sync %0, 64;" ::"n"(kBarIssue) : "memory");
        bool ok = s_first_ok != 0;
        if (ok) {
          tc_fence_after();
          if (elect_one()) issue_s(0);
          __syncwarp();
        }
        if (n_kv > 1) {
          __syncwarp();
          asm volatile("bar.sync %0, 64;" ::"n"(kBarIssue) : "memory");
          ok = ok && s_second_ok != 0;
          if (ok) {
            tc_fence_after();
            if (elect_one()) issue_s(1);
            __syncwarp();
          }
        }
        for (int j = 0; j < n_kv; ++j) {
          __syncwarp();
          asm volatile("bar.sync %0, %1;" ::"n"(kBarRound), "n"(kRoundThreads) : "memory");
          ok = ok && s_round_ok[j & 1] != 0 && !*abort_flag;
          if (!ok) continue;
          tc_fence_after();
          // O_h += P_{j,h} V_{j,h} for both halves h, then S_{j+2} into the same buffer
          // (executed after this P V, which reads P_j from it).
          const int b = j & 1, st = j % kVStages;
          const uint64_t dv = dv0 + (uint64_t)((st * kKVBytes) >> 4);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
          if (elect_one()) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int ks = 0; ks < kHalf / 16; ++ks)
                mma_ts(tmem + col_o(h, D), tmem + col_s(b, h) + ks * 8,
                       dv + (uint64_t)(((h * (kHalf / 16) + ks) * 16 * 128) >> 4), idesc_o, ks > 0 ? 1u : acc0);
            }
            tc_commit(smem_u32(&bars.pv_done[st]));
            if (j + 2 < n_kv) issue_s(j + 2);
          }
          __syncwarp();
        }
        // All tensor-core work issued by this CTA completes before TMEM is freed.
        if (elect_one()) tc_commit(smem_u32(&bars.drain));
        __syncwarp();
        mbar_wait(smem_u32(&bars.drain), 0, abort_flag, p.err, 14, false, kLimit);
      }
    }
    __syncwarp();
  } else {
    const int wg = warp / 4;  // this warpgroup takes keys [64 wg, 64 wg + 64) of every key tile
    const int r = threadIdx.x % kBM;
    const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    // m_ref: reference max (log2 units) that this warpgroup's O and l are scaled to.
    float m_ref = -INFINITY, l = 0.0f;
    bool ok = true;
    // counting instance: weights below eps are the scores below tau = max + log2(eps * sum)
    float tau = 0.0f;
    int cnt = 0;
    if constexpr (COUNT) {
      const int t = min(t0 + r / p.group, t_last);
      const float2 st = p.count_stats[(size_t)t * p.hq + (size_t)g * p.group + (r % p.group)];
      tau = st.x + p.log2_eps + __log2f(st.y);
    }
    // Wait until P V_j is complete (barrier pv_done[j % 3], its phase j / 3). Polled: a
    // suspended waiter resumes late, and these waits sit on the tile loop's critical path.
    auto wait_pv = [&](int j, int site) -> bool {
      const bool w =
          mbar_spin(smem_u32(&bars.pv_done[j % kVStages]), (j / kVStages) & 1, abort_flag, p.err, site, kLimit);
      return __all_sync(0xffffffffu, w);
    };
    // One tile; false if a wait gave up (the abort flag is raised then).
    auto tile = [&](int j) -> bool {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu,
                      mbar_spin(smem_u32(&bars.s_done[j % kKStages]), (j / kKStages) & 1, abort_flag, p.err, 20 + wg,
                                kLimit)))
        return false;
      tc_fence_after();
      // Copy this half's 64 scores to registers; P_j is later written over their first 32 columns.
      uint32_t sv[kHalf];
      {
        uint32_t(&sa)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t(&sb)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tmem_ld_x32_async(lane_base + col_s(b, wg), sa);
        tmem_ld_x32_async(lane_base + col_s(b, wg) + 32, sb);
        tmem_wait_ld(sa);
        tmem_wait_ld(sb);
      }
      const int lim = my_pos - (j * kBN + wg * kHalf);  // columns c <= lim are visible to this row
      const bool diag = __any_sync(0xffffffffu, lim < kHalf - 1);  // diagonal tiles only
      if (diag) {
#pragma unroll
        for (int c = 0; c < kHalf; ++c)
          if (c > lim) sv[c] = 0xff800000u;  // -inf
      }
      if constexpr (COUNT) {  // masked columns (-inf) count too; the epilogue corrects for the tile edge
#pragma unroll
        for (int c = 0; c < kHalf; ++c) cnt += __uint_as_float(sv[c]) * p.scale_log2 < tau ? 1 : 0;
      }

      // P = 2^(s * scale - m_ref), packed to bf16, and its row sum. A row's first visible tile sets
      // the reference m_ref (log2 units) that O and l are scaled to: the max of its scores. Later
      // tiles run the exponentials against the reference without taking their max first (the
      // softmax is on the tile loop's critical path): a half tile whose row sum stays within 2^16
      // has every P within 2^16, far from overflow in P, O and l. One whose sum passes that (its
      // max grew by more than 2^10) takes its max, moves the reference of the rows whose max passes
      // it by more than 2^8, rescales O and computes P again (from the scores loaded again: S is
      // still in TMEM, since P is stored over it only at the end, and the registers are not kept).
      // A row with nothing visible yet has only -inf scores, so P = 0 (the offset 0 stands in for
      // its missing reference).
      uint32_t pk[kHalf / 2];
      bool move_ref = !__all_sync(0xffffffffu, m_ref != -INFINITY);
      float sum = 0.0f;
      if (!move_ref) {
        sum = softmax_p(sv, m_ref, p.scale_log2, pk);
        if (!__all_sync(0xffffffffu, sum <= kTileSumLimit)) {  // rare: the max jumped
          move_ref = true;
          uint32_t(&sa)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t(&sb)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          tmem_ld_x32_async(lane_base + col_s(b, wg), sa);
          tmem_ld_x32_async(lane_base + col_s(b, wg) + 32, sb);
          tmem_wait_ld(sa);
          tmem_wait_ld(sb);
          if (diag) {
#pragma unroll
            for (int c = 0; c < kHalf; ++c)
              if (c > lim) sv[c] = 0xff800000u;  // -inf
          }
        }
      }
      if (move_ref) {
        // Four independent chains of three-input max (8 deep each).
        float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kHalf; c += 8) {
          tm[0] = max3(tm[0], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
          tm[1] = max3(tm[1], __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
          tm[2] = max3(tm[2], __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
          tm[3] = max3(tm[3], __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
        }
        const float mt = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])) * p.scale_log2;  // -inf: nothing visible
        const bool up = mt > m_ref + kRescaleThreshold;  // always, at a row's first visible key
        if (__any_sync(0xffffffffu, up)) {
          // alpha = 2^(m_ref - mt): 0 for a row that had nothing visible (its O and l are zero).
          const float alpha = up ? ex2(m_ref - mt) : 1.0f;
          const bool scale_o = up && m_ref != -INFINITY;
          if (up) {
            l *= alpha;
            m_ref = mt;
          }
          // O holds this warpgroup's sum through tile j - 1: wait for that P V, then scale it.
          if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
            if (!wait_pv(j - 1, 22 + wg)) return false;
            tc_fence_after();
            const float a = scale_o ? alpha : 1.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld_x32(lane_base + col_o(wg, D) + c0, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
              tmem_st_x32(lane_base + col_o(wg, D) + c0, o);
            }
            tmem_st_wait();
          }
        }
        sum = softmax_p(sv, m_ref, p.scale_log2, pk);
      }
      l += sum;
      tmem_st_x32(lane_base + col_s(b, wg), pk);
      tmem_st_wait();
      return true;
    };
    // Every softmax warp syncs on kBarRound once per key tile, also after a failed wait (then
    // without work), so every round of the issuer and its waiter completes. A blocking sync, not
    // an arrival: a warp cannot reach the next round's barrier before this round's has completed,
    // so no arrival is ever counted in the wrong round. It costs little: the next tile needs
    // S_{j+1}, which the issuer finishes issuing just before it joins this barrier.
    for (int j = 0; j < n_kv; ++j) {
      if (ok) ok = tile(j);
      tc_fence_before();
      __syncwarp();
      asm volatile("bar.sync %0, %1;" ::"n"(kBarRound), "n"(kRoundThreads) : "memory");
    }
    if (ok) ok = wait_pv(n_kv - 1, 26 + wg);
    // Merge the two warpgroups' partial results; each writes half of the columns.
    // [warpgroup][max, sum][row] in the K ring: every K tile has been consumed by now (the last
    // P V is complete and the S MMAs before it), so the ring is free.
    float(*s_ml)[2][kBM] = reinterpret_cast<float(*)[2][kBM]>(smem_raw + (sK0 - smem_u32(smem_raw)));
    // the output's staging boxes in the V ring, also free now (the last P V has completed)
    constexpr uint32_t kOutBox = kBM * 128;
    const uint32_t sOut = sV0;
    int(*s_cnt)[kBM] = reinterpret_cast<int(*)[kBM]>(smem_raw + (sK0 - smem_u32(smem_raw)) + 4 * kBM * 4);
    s_ml[wg][0][r] = m_ref;
    s_ml[wg][1][r] = l;
    if constexpr (COUNT) s_cnt[wg][r] = cnt;
    tc_fence_before();
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(2 * kSoftmaxThreads) : "memory");
    ok = ok && !*abort_flag;
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float m0 = s_ml[0][0][r], m1 = s_ml[1][0][r];
      const float mm = fmaxf(m0, m1);
      const float a0 = m0 == -INFINITY ? 0.0f : ex2(m0 - mm);
      const float a1 = m1 == -INFINITY ? 0.0f : ex2(m1 - mm);
      const float sum = s_ml[0][1][r] * a0 + s_ml[1][1][r] * a1;
      const float inv = 1.0f / sum;
      const int t = t0 + r / p.group;
      const bool valid = t <= t_last;
      const size_t row = (size_t)t * p.hq + (size_t)g * p.group + (r % p.group);
      if (valid && p.row_stats != nullptr) p.row_stats[row] = make_float2(mm, sum);
      // the visited tiles cover keys [0, 128 n_kv): keys past n_keys were counted as masked,
      // keys past the last visited tile were not visited and are all masked for this row
      if constexpr (COUNT)
        if (valid) p.counts[row] = s_cnt[0][r] + s_cnt[1][r] + (p.n_keys - n_kv * kBN);
      // out = O_0 (a_0 / sum) + O_1 (a_1 / sum): both chunks' loads issued before one wait
      const float b0 = a0 * inv, b1 = a1 * inv;
      constexpr int kChunks = (D / 2) / 32;
      uint32_t o0[kChunks][32], o1[kChunks][32];
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        tmem_ld_x32_async(lane_base + col_o(0, D) + wg * (D / 2) + ch * 32, o0[ch]);
        tmem_ld_x32_async(lane_base + col_o(1, D) + wg * (D / 2) + ch * 32, o1[ch]);
      }
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        tmem_wait_ld(o0[ch]);
        tmem_wait_ld(o1[ch]);
      }
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            f[e] = fmaf(__uint_as_float(o0[ch][q * 8 + e]), b0, __uint_as_float(o1[ch][q * 8 + e]) * b1);
          const int c = wg * (D / 2) + ch * 32 + q * 8;
          const uint4 pk = pack8(f);
          // row r of the output box holding columns c: 128-byte rows, 16-byte chunks swizzled
          const uint32_t dst = sOut + (uint32_t)(c / 64) * kOutBox + (uint32_t)r * 128u +
                               (uint32_t)((((c % 64) / 8) ^ (r & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk.x), "r"(pk.y), "r"(pk.z),
                       "r"(pk.w)
                       : "memory");
        }
      }
    }
    // The tile's rows are one box of the output (TQ tokens x G heads x 64 columns, as Q was loaded):
    // one TMA store per 64 columns; rows past mq are clipped by the tensor map.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(2 * kSoftmaxThreads) : "memory");
    if (threadIdx.x == 0 && !*abort_flag) {
#pragma unroll
      for (int b = 0; b < kBoxes; ++b)
        asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                         &tm_o),
                     "r"(b * 64), "r"(0), "r"(g), "r"(t0), "r"(sOut + b * kOutBox)
                     : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the box has left shared memory
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int D, bool COUNT, bool PROBE = false>
cudaError_t launch_typed(const void* q, QueryPositions qp, int mq, const void* k, const void* v, int n_keys,
                         int hq, int hkv, float scale, void* out, const AttentionDiag& diag, int32_t* err,
                         cudaStream_t s) {
  const int group = hq / hkv;
  const int tq = kBM / group;
  const int n_qtiles = (mq + tq - 1) / tq;
  CUtensorMap tq_map, tk_map, tv_map, to_map;
  const cuuint64_t qd[4] = {(cuuint64_t)D, (cuuint64_t)group, (cuuint64_t)hkv, (cuuint64_t)mq};
  const cuuint64_t qs[3] = {(cuuint64_t)D * 2, (cuuint64_t)group * D * 2, (cuuint64_t)hq * D * 2};
  const cuuint32_t qb[4] = {64, (cuuint32_t)group, 1, (cuuint32_t)tq};
  const cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)n_keys};
  const cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
  const cuuint32_t kbx[3] = {64, 1, (cuuint32_t)kBN};  // a K or V tile: kBN keys of one kv head
  if (!encode_map(&tq_map, q, 4, qd, qs, qb) || !encode_map(&tk_map, k, 3, kd, ks, kbx) ||
      !encode_map(&tv_map, v, 3, kd, ks, kbx) || !encode_map(&to_map, out, 4, qd, qs, qb))
    return cudaErrorInvalidValue;
  Params p;
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
  p.n_qtiles = n_qtiles;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = static_cast<uint8_t*>(out);
  p.err = err;
  p.row_stats = diag.row_stats;
  p.count_stats = diag.count_stats;
  p.log2_eps = diag.log2_eps;
  p.counts = diag.counts;
  size_t smem = 1024 + (size_t)(kBM + (kKStages + kVStages) * kBN) * D * 2;
  if (smem < 117 * 1024) smem = 117 * 1024;  // one CTA per SM: the CTA takes all 512 TMEM columns
  static std::atomic<uint64_t> configured{0};
  const cudaError_t e = set_smem_limit_once(hkvd_attention_kernel<D, COUNT, PROBE>, (int)smem, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(hkvd_attention_kernel<D, COUNT, PROBE>, n_qtiles * hkv, kThreads, smem, s, tq_map, tk_map,
                    tv_map, to_map, p);
}

}  // namespace

cudaError_t launch_hkvd_attention(const void* q, QueryPositions qp, int32_t mq, const void* k, const void* v,
                                  int32_t n_keys, int32_t hq, int32_t hkv, int32_t head_dim, float scale, void* out,
                                  int32_t* err, cudaStream_t s, const AttentionDiag& diag) {
  if (mq <= 0) return cudaSuccess;
  const bool count = diag.counts != nullptr;
  if (!count && diag.row_stats == nullptr && attention_pp_eligible(mq, hq, hkv, head_dim)) {
    const cudaError_t e = launch_hkvd_attention_pp(q, qp, mq, k, v, n_keys, hq, hkv, scale, out, err, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (head_dim == 128)
    return count ? launch_typed<128, true>(q, qp, mq, k, v, n_keys, hq, hkv, scale, out, diag, err, s)
                 : launch_typed<128, false>(q, qp, mq, k, v, n_keys, hq, hkv, scale, out, diag, err, s);
  if (head_dim == 64)
    return count ? launch_typed<64, true>(q, qp, mq, k, v, n_keys, hq, hkv, scale, out, diag, err, s)
                 : launch_typed<64, false>(q, qp, mq, k, v, n_keys, hq, hkv, scale, out, diag, err, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_timeout_probe(const void* q, QueryPositions qp, int32_t mq, const void* k,
                                           const void* v, int32_t n_keys, int32_t hq, int32_t hkv, float scale,
                                           void* out, int32_t* err, cudaStream_t s) {
  if (mq <= 0 || n_keys <= kBN) return cudaErrorInvalidValue;
  return launch_typed<128, false, true>(q, qp, mq, k, v, n_keys, hq, hkv, scale, out, AttentionDiag(), err, s);
}

}  // namespace cb
