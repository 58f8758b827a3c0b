// Blockwise packed attention on CTA pairs (tcgen05 cta_group::2, sm_103a).
//
// The same computation as the one-CTA kernel in attn_tc.cu, one "partial
// attention" step (HSAP abstract) per 128-key tile merged into the running
// (O, LSE) by the log-sum-exp rule (TASP abstract), with the same masks.
// What changes is how the work is laid over the SMs. Two CTAs of a cluster
// (one per SM of a pair) take two query heads that share a key/value head
// (GQA), over the same 256 rows. Their rows see the same documents and the
// same causal limits, so both walk the same key tiles. Each tensor-core
// instruction is a 256-row MMA: rows 0-127 are the first CTA's query head and
// rows 128-255 the second's. The B operand (K for S = Q K^T, V for O += P V)
// is split between the two CTAs' shared memory: the first holds keys 0-63 of
// a K tile and dims 0-63 of a V tile, the second the other halves. Each SM
// thus reads half a K/V tile per MMA from its own shared memory instead of a
// whole one and loads half of each tile (160 KB of shared-memory traffic per
// key tile instead of 256 KB). Measured on the 32K-token layer, the MMAs take
// as long as in the one-CTA kernel; what the pair gains is a shorter softmax
// hand-off, and the freed shared memory holds a second Q buffer.
//
// Roles (12 warps per CTA):
//   warp 0      TMA producer, in both CTAs: Q tiles of the CTA's head (two
//               buffers: the next unit's Q loads during the current unit), and
//               the CTA's halves of K (2 stages) and V (3 stages). Copies are
//               counted on the first CTA's barriers.
//   warp 1      allocates tensor memory (both CTAs); in the first CTA, lane 0
//               issues every MMA of the pair and signals both CTAs.
//   warp 2      in the first CTA, lane 0 claims the work units and publishes
//               each unit's record (rows, Q tiles, documents, the cursor on
//               its first tile) to both CTAs, up to two units ahead.
//   warps 4-11  softmax for Q tile 0 / 1 of the CTA's head, as in attn_tc.cu.
// Tensor memory per CTA: S_i at 128 i, P_i in columns [64, 128) of S_i, O_i at
// 256 + 128 i. The MMA order per tile is QK0(j), PV1(j-1), QK1(j), PV0(j).

#include <cuda.h>

#include <mutex>

#include "sp_device.cuh"
#include "sp_tiles.cuh"

namespace sp {
namespace {

constexpr int REC_TILE = 16, REC_LAST = 32;

struct PCfg {
  static constexpr int D = 128;
  // Two Q buffers (the next unit's Q tiles load while the current unit runs),
  // three K and three V stages (V is held one MMA group longer than K): copies
  // run two tiles ahead (with two K stages, one: 0.3-0.6% slower).
  static constexpr int QBUF = 2;
  static constexpr int KSTAGE = 3;
  static constexpr int VSTAGE = 3;
  static constexpr int Q_SUB = 128 * 128;           // [128 rows][64 dims] bf16
  static constexpr int Q_TILE = 2 * Q_SUB;          // 128 rows x 128 dims
  static constexpr int K_SUB = 64 * 128;            // [64 keys][64 dims]
  static constexpr int K_STAGE_BYTES = 2 * K_SUB;   // half a K tile: 64 keys x 128 dims
  static constexpr int V_STAGE_BYTES = 128 * 128;   // half a V tile: 128 keys x 64 dims
  static constexpr int Q_BUF_BYTES = 2 * Q_TILE;   // the unit's two Q tiles
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QBUF * Q_BUF_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGE * K_STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_V + VSTAGE * V_STAGE_BYTES;
  static constexpr int N_BARS = 24;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;   // TMEM address, abort flag
  static constexpr int OFF_REC = OFF_MISC + 8;
  static constexpr int OFF_URING = (OFF_REC + 4 * KSTAGE + 15) & ~15;  // two unit records
  static constexpr int SMEM_ALLOC = OFF_URING + 2 * 128 + 1024;  // 230,880 of 232,448 bytes
  static constexpr int TM_S = 0;
  static constexpr int TM_O = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(256, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(256, D, 0, 1);
  // Bytes one tile's copies bring to the pair: both CTAs' K and V halves.
  static constexpr uint32_t KV_TX = 2 * (K_STAGE_BYTES + V_STAGE_BYTES);
  static constexpr uint32_t Q_TX = 2 * 2 * Q_TILE;
};

// Barrier slots. The full barriers (Q_FULL, KV_FULL), P_FULL and U_EMPTY are
// used in the first CTA only; the others exist in both CTAs and receive the
// MMA lane's multicast commits. Q_FULL / Q_EMPTY: one per Q buffer.
enum {
  B_Q_FULL = 0, B_Q_EMPTY = 2, B_KV_FULL = 4, B_K_EMPTY = 7, B_V_EMPTY = 10,
  B_S_FULL = 13, B_P_FULL = 15, B_O_FULL = 17, B_DRAIN = 19, B_U_FULL = 20, B_U_EMPTY = 22
};
static_assert(B_U_EMPTY + 2 <= PCfg::N_BARS, "barrier slots");
static_assert(PCfg::SMEM_ALLOC <= 232448, "pair kernel layout exceeds the shared memory of a block");

// A unit slot holds the unit's record (sp_tiles.cuh), built by the first CTA's
// scheduler warp and stored into both CTAs' slot. Both CTAs' units have the
// same rows, documents and items; the second CTA's query head is the first's
// plus one.

// Consumers of a unit slot: the producer, the MMA lane and 8 softmax warps of
// the first CTA, the producer and 8 softmax warps of the second.
constexpr int UNIT_CONSUMERS = 19;
// Softmax warps of both CTAs storing P_i.
constexpr int P_ARRIVALS = 8;

// ------------------------------------------------------------ cluster PTX

// TMA load into this CTA's shared memory whose completion is counted on a
// barrier of either CTA of the pair (cl_bar: cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, uint32_t cl_bar, int x,
                                                 int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(tmap), "r"(cl_bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols)
               : "memory");
}
// Arrives on the barrier at this offset in both CTAs once every MMA issued so
// far by this thread has completed.
__device__ __forceinline__ void commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      :: "r"(bar), "h"(static_cast<uint16_t>(3)) : "memory");
}
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Probe {
  uint32_t bar, par;
  int on;
};

__device__ __forceinline__ int run_probes(const Probe& a, const Probe& b) {
  int r = 0;
  if (a.on && mbar_test(a.bar, a.par)) r |= 1;
  if (b.on && mbar_test(b.bar, b.par)) r |= 2;
  return r;
}

// S = Q K^T for Q tile i of both heads: 8 MMAs of 256x128x16. A (Q) advances
// 32 bytes per K step inside a 128-row sub-tile; B (the CTA's 64 keys of K)
// inside a 64-row sub-tile.
__device__ __forceinline__ int mma_qk(uint32_t d_t, uint64_t a0, uint64_t b0, const Probe& pa,
                                      const Probe& pb) {
  using C = PCfg;
  int res = 0;
#pragma unroll
  for (int kk = 0; kk < C::D / 16; ++kk) {
    if (kk == C::D / 16 - 1) res = run_probes(pa, pb);
    const uint64_t ao = static_cast<uint64_t>(((kk >> 2) * C::Q_SUB + (kk & 3) * 32) >> 4);
    const uint64_t bo = static_cast<uint64_t>(((kk >> 2) * C::K_SUB + (kk & 3) * 32) >> 4);
    mma_ss_pair(d_t, a0 + ao, b0 + bo, C::IDESC_QK, kk > 0 ? 1u : 0u);
  }
  return res;
}

// Half h of O += P V: keys 64h .. 64h+63; P from tensor memory, the CTA's 64
// dims of V from shared memory (MN-major, 16 keys = 2048 bytes per K step).
__device__ __forceinline__ int mma_pv_half(uint32_t d_t, uint32_t a_t, uint64_t b0, int h, int acc,
                                           const Probe& pa, const Probe& pb) {
  using C = PCfg;
  int res = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kk = 4 * h + q;
    if (q == 3) res = run_probes(pa, pb);
    mma_ts_pair(d_t, a_t + 8 * kk, b0 + static_cast<uint64_t>(kk * (2048 >> 4)), C::IDESC_PV,
                (acc || kk > 0) ? 1u : 0u);
  }
  return res;
}

template <int OUT_FP32>
__global__ void __launch_bounds__(384, 1)
attn_tc_pair_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using C = PCfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  // The dynamic shared memory starts at the same offset in both CTAs, so
  // every buffer and barrier has the same address in each.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* rec = reinterpret_cast<volatile int*>(smem + C::OFF_REC);
  volatile int* uring = reinterpret_cast<volatile int*>(smem + C::OFF_URING);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();
  const bool lead = rank == 0;

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::QBUF; ++b) {
      mbar_init(bar(B_Q_FULL + b), 1);
      mbar_init(bar(B_Q_EMPTY + b), 1);
    }
    for (int s = 0; s < C::KSTAGE; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::VSTAGE; ++s) mbar_init(bar(B_V_EMPTY + s), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_P_FULL + i), P_ARRIVALS);
      mbar_init(bar(B_O_FULL + i), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_U_FULL + i), 1);
      mbar_init(bar(B_U_EMPTY + i), UNIT_CONSUMERS);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // Barriers of both CTAs are initialised before either CTA touches the other's.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_pairs = n_units_of(a) >> 1;
  const int G = a.Hq / a.Hkv;
  const unsigned long long tmo = a.timeout_ns;
  // Barriers and unit slots of the first CTA, as cluster addresses.
  const uint32_t lead_bar0 = map_to(bar0, 0);
  auto lbar = [&](int i) { return lead_bar0 + 8u * static_cast<uint32_t>(i); };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 136;");
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      uint32_t unit_cnt = 0;
      int kst = 0, vst = 0;
      uint32_t kph = 0, vph = 0;
      int armed_k[C::KSTAGE] = {};
      uint32_t par_k[C::KSTAGE] = {};
      int armed_q[C::QBUF] = {};
      uint32_t par_q[C::QBUF] = {};
      bool ok = true;
      int uslot = 0;
      uint32_t uph = 0;
      for (;; ++unit_cnt) {
        int h = 0, q0 = 0;
        QTile qt[2];
        Cursor cur;
        bool have = false;
        int ka = 0, kb = 0, cls[2] = {0, 0};
        const volatile int* rs = uring + UREC_WORDS * uslot;
        if (!wait_cl(bar(B_U_FULL + uslot), uph, tmo, a.err, abort_flag)) { ok = false; break; }
        const int v = rs[UR_V];
        if (v >= 0) read_unit_record(rs, static_cast<int>(rank), h, q0, qt, cur);
        arrive_cluster(lbar(B_U_EMPTY + uslot));
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (v < 0) break;
        have = next_tile(a, cur, qt, ka, kb, cls);
        const int hk = h / G;
        const int qb = unit_cnt & 1;
        const uint32_t qph = (unit_cnt >> 1) & 1;
        if (!mbar_wait_bounded(bar(B_Q_EMPTY + qb), qph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
        if (lead) {
          mbar_arrive_expect_tx(bar(B_Q_FULL + qb), C::Q_TX);
          armed_q[qb] = 1;
          par_q[qb] = qph;
        }
        for (int i = 0; i < 2; ++i)
          for (int s = 0; s < 2; ++s)
            tma_load_3d_pair(sQ + qb * C::Q_BUF_BYTES + i * C::Q_TILE + s * C::Q_SUB, &tmq,
                             lbar(B_Q_FULL + qb), 64 * s, h, q0 + 128 * i);
        if (!have) {
          if (!mbar_wait_bounded(bar(B_K_EMPTY + kst), kph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
          if (lead) {
            rec[kst] = REC_LAST;
            mbar_arrive(bar(B_KV_FULL + kst));
          }
          if (++kst == C::KSTAGE) { kst = 0; kph ^= 1; }
        }
        while (have) {
          int nka, nkb, ncls[2];
          const bool nxt = next_tile(a, cur, qt, nka, nkb, ncls);
          if (!mbar_wait_bounded(bar(B_K_EMPTY + kst), kph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
          if (!mbar_wait_bounded(bar(B_V_EMPTY + vst), vph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
          if (lead) {
            rec[kst] = REC_TILE | cls[0] | (cls[1] << 2) | (nxt ? 0 : REC_LAST);
            mbar_arrive_expect_tx(bar(B_KV_FULL + kst), C::KV_TX);
            armed_k[kst] = 1;
            par_k[kst] = kph;
          }
          const uint32_t full = lbar(B_KV_FULL + kst);
          // This CTA's 64 keys of the K tile; a box wholly past the last token
          // starts at the last token instead (its columns are masked).
          const int krow = min(ka + 64 * static_cast<int>(rank), a.T - 1);
          for (int s = 0; s < 2; ++s)
            tma_load_3d_pair(sK + kst * C::K_STAGE_BYTES + s * C::K_SUB, &tmk, full, 64 * s, hk, krow);
          tma_load_3d_pair(sV + vst * C::V_STAGE_BYTES, &tmv, full, 64 * static_cast<int>(rank), hk, ka);
          if (++kst == C::KSTAGE) { kst = 0; kph ^= 1; }
          if (++vst == C::VSTAGE) { vst = 0; vph ^= 1; }
          ka = nka;
          kb = nkb;
          cls[0] = ncls[0];
          cls[1] = ncls[1];
          have = nxt;
        }
        if (!ok) break;
      }
      if (!ok) {
        // Aborting: let the copies already issued land before the CTA leaves.
        // The first CTA waits for its armed phases; the second cannot wait on
        // the first CTA's barriers and gives its copies a fixed time.
        volatile int no_abort = 0;
        const unsigned long long drain = 50000000ull;
        if (lead) {
          for (int b = 0; b < C::QBUF; ++b)
            if (armed_q[b]) mbar_wait_bounded(bar(B_Q_FULL + b), par_q[b], drain, a.err, &no_abort);
          for (int s = 0; s < C::KSTAGE; ++s)
            if (armed_k[s]) mbar_wait_bounded(bar(B_KV_FULL + s), par_k[s], drain, a.err, &no_abort);
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < drain) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ unit scheduler (first CTA)
    if (lead && lane == 0) {
      int k_static = 0;
      auto fetch = [&]() -> int {
        int v;
        if (a.work_counter) {
          v = atomicAdd(a.work_counter, 1);
        } else {
          v = static_cast<int>(cluster_idx()) + k_static * static_cast<int>(n_clusters());
          ++k_static;
        }
        return v < n_pairs ? v : -1;
      };
      const uint32_t peer_uring = map_to(smem_u32(const_cast<int*>(uring)), 1);
      const uint32_t peer_ufull = map_to(bar(B_U_FULL), 1);
      int uslot = 0;
      uint32_t uph = 0;
      for (;;) {
        // The record is built before the slot is free: its table searches and
        // the walk to the first tile overlap the other roles' work.
        const int v = fetch();
        int w[UR_N];
        w[UR_V] = v;
        if (v >= 0) build_unit_record(a, 2 * v, v, w);
        if (!wait_cl(bar(B_U_EMPTY + uslot), uph ^ 1, tmo, a.err, abort_flag)) break;
        volatile int* rs = uring + UREC_WORDS * uslot;
        const int n = v >= 0 ? static_cast<int>(UR_N) : 1;
        const uint32_t prs = peer_uring + 4u * UREC_WORDS * uslot;
        for (int i = 0; i < n; ++i) {
          rs[i] = w[i];
          st_cluster(prs + 4u * i, w[i]);
        }
        mbar_arrive(bar(B_U_FULL + uslot));
        arrive_cluster(peer_ufull + 8u * uslot);
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (v < 0) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (first CTA)
    if (lead && lane == 0) {
      const uint64_t dq00 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dq01 = smem_desc_sw128(sQ + C::Q_TILE, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sV, C::V_STAGE_BYTES, 1024);
      uint32_t unit_cnt = 0, pcnt0 = 0, pcnt1 = 0;
      int kst = 0, vst = 0;
      uint32_t kph = 0;
      bool ok = true;
      const Probe none{0u, 0u, 0};
      const uint32_t dS0 = tmem + C::TM_S, dS1 = tmem + C::TM_S + 128;
      const uint32_t dO0 = tmem + C::TM_O, dO1 = tmem + C::TM_O + D;
      const uint32_t aP0 = dS0 + 64, aP1 = dS1 + 64;
      const uint64_t kstep = C::K_STAGE_BYTES >> 4;
      const uint64_t vstep = C::V_STAGE_BYTES >> 4;

      bool rdy_k = false;
      int uslot = 0;
      uint32_t uph = 0;
      for (;; ++unit_cnt) {
        if (!wait_cl(bar(B_U_FULL + uslot), uph, tmo, a.err, abort_flag)) { ok = false; break; }
        const int v = uring[UREC_WORDS * uslot + UR_V];
        mbar_arrive(bar(B_U_EMPTY + uslot));
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (v < 0) break;
        const int qb = unit_cnt & 1;
        if (!mbar_wait_bounded(bar(B_Q_FULL + qb), (unit_cnt >> 1) & 1, tmo, a.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t qoff = static_cast<uint64_t>((qb * C::Q_BUF_BYTES) >> 4);
        const uint64_t dq0 = dq00 + qoff, dq1 = dq01 + qoff;
        int has_pv0 = 0, has_pv1 = 0;
        int have_prev = 0, prev_vs = 0, prev_c1 = 0;
        while (true) {
          if (!rdy_k && !mbar_wait_bounded(bar(B_KV_FULL + kst), kph, tmo, a.err, abort_flag)) { ok = false; break; }
          rdy_k = false;
          tc_fence_after();
          const int r = rec[kst];
          const int nkst = (kst + 1 == C::KSTAGE) ? 0 : kst + 1;
          const uint32_t nkph = (kst + 1 == C::KSTAGE) ? (kph ^ 1) : kph;
          if (r & REC_TILE) {
            const int c0 = r & 3, c1 = (r >> 2) & 3;
            const int pv1 = have_prev && prev_c1 != CLS_SKIP;
            const uint64_t bK = dk0 + static_cast<uint64_t>(kst) * kstep;
            const uint64_t bV = dv0 + static_cast<uint64_t>(vst) * vstep;
            const uint64_t bVp = dv0 + static_cast<uint64_t>(prev_vs) * vstep;
            const Probe p1{bar(B_P_FULL + 1), pcnt1 & 1, pv1};
            const Probe p0{bar(B_P_FULL + 0), pcnt0 & 1, c0 != CLS_SKIP};
            const Probe pk{bar(B_KV_FULL + nkst), nkph, 1};
            int got1 = 0, got0 = 0;
            if (c0 != CLS_SKIP) {
              got1 = mma_qk(dS0, dq0, bK, p1, none) & 1;
              commit_both(bar(B_S_FULL + 0));
            }
            if (pv1) {
              if (!got1 && !mbar_wait_bounded(p1.bar, p1.par, tmo, a.err, abort_flag)) { ok = false; break; }
              tc_fence_after();
              mma_pv_half(dO1, aP1, bVp, 0, has_pv1, none, none);
              got0 = mma_pv_half(dO1, aP1, bVp, 1, 1, p0, none) & 1;
              ++pcnt1;
              has_pv1 = 1;
            }
            if (have_prev) commit_both(bar(B_V_EMPTY + prev_vs));
            if (c1 != CLS_SKIP) {
              const int g = mma_qk(dS1, dq1, bK, got0 ? none : p0, none);
              got0 |= g & 1;
              commit_both(bar(B_S_FULL + 1));
            }
            commit_both(bar(B_K_EMPTY + kst));
            if (c0 != CLS_SKIP) {
              if (!got0 && !mbar_wait_bounded(p0.bar, p0.par, tmo, a.err, abort_flag)) { ok = false; break; }
              tc_fence_after();
              mma_pv_half(dO0, aP0, bV, 0, has_pv0, none, none);
              rdy_k = mma_pv_half(dO0, aP0, bV, 1, 1, (r & REC_LAST) ? none : pk, none) & 1;
              ++pcnt0;
              has_pv0 = 1;
            }
            have_prev = 1;
            prev_vs = vst;
            prev_c1 = c1;
            if (++vst == C::VSTAGE) vst = 0;
          } else {
            commit_both(bar(B_K_EMPTY + kst));
          }
          kst = nkst;
          kph = nkph;
          if (r & REC_LAST) break;
        }
        if (!ok) break;
        // O_0 is complete once the PV0 issued so far are: the softmax warps of Q
        // tile 0 may read it out while the last PV1 still waits for its P.
        commit_both(bar(B_O_FULL + 0));
        if (have_prev) {
          if (prev_c1 != CLS_SKIP) {
            const uint64_t bVp = dv0 + static_cast<uint64_t>(prev_vs) * vstep;
            if (!mbar_wait_bounded(bar(B_P_FULL + 1), pcnt1 & 1, tmo, a.err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            mma_pv_half(dO1, aP1, bVp, 0, has_pv1, none, none);
            mma_pv_half(dO1, aP1, bVp, 1, 1, none, none);
            ++pcnt1;
          }
          commit_both(bar(B_V_EMPTY + prev_vs));
        }
        commit_both(bar(B_Q_EMPTY + qb));
        commit_both(bar(B_O_FULL + 1));
      }
      // Every MMA issued has completed before tensor memory is released.
      volatile int no_abort = 0;
      commit_both(bar(B_DRAIN));
      mbar_wait_bounded(bar(B_DRAIN), 0, 50000000ull, a.err, &no_abort);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    const int wg = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + 128 * wg;
    const uint32_t tO = tmem + lane_off + C::TM_O + D * wg;
    const float sl2 = a.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const uint32_t p_full = lbar(B_P_FULL + wg);
    // O rows start 32-byte aligned when the output does (rows are 256 or 512 bytes).
    const bool o_a32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
    uint32_t s_cnt = 0, unit_cnt = 0;
    bool ok = true;
    int uslot = 0;
    uint32_t uph = 0;
    for (;; ++unit_cnt) {
      if (!wait_cl(bar(B_U_FULL + uslot), uph, tmo, a.err, abort_flag)) { ok = false; break; }
      const volatile int* rs = uring + UREC_WORDS * uslot;
      const int v = rs[UR_V];
      int h = 0, q0 = 0;
      QTile qt[2];
      Cursor cur;
      if (v >= 0) read_unit_record(rs, static_cast<int>(rank), h, q0, qt, cur);
      __syncwarp();
      if (lane == 0) arrive_cluster(lbar(B_U_EMPTY + uslot));
      if (++uslot == 2) { uslot = 0; uph ^= 1; }
      if (v < 0) break;
      const QTile my = wg ? qt[1] : qt[0];
      const int t = q0 + 128 * wg + r;
      const bool valid = (t >= my.qa) && (t < my.qb);
      int rds = 0, rde = 0;
      if (valid) {
        if (my.one_doc) {  // the tile's rows are all in one document
          rds = my.ds;
          rde = my.de;
        } else {
          const int dd = doc_of(a.cu, a.ndocs, t);
          rds = __ldg(a.cu + dd);
          rde = __ldg(a.cu + dd + 1);
        }
      }
      const int rcausal_end = a.causal ? t + 1 : 0x7fffffff;
      float m = NEG_INF, l = 0.f;
      int has_pv = 0;
      int ka, kb, cls[2];
      while (next_tile(a, cur, qt, ka, kb, cls)) {
        const int c = wg ? cls[1] : cls[0];
        if (c == CLS_SKIP) continue;
        if (!mbar_wait_bounded(bar(B_S_FULL + wg), s_cnt & 1, tmo, a.err, abort_flag)) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128_sync(tS, sr);
        if (c == CLS_MASKED) {
          int lo = 0, hi = 0;
          if (valid) {
            lo = max(ka, rds) - ka;
            hi = min(min(kb, rde), rcausal_end) - ka;
          }
#pragma unroll
          for (int j = 0; j < 128; ++j)
            sr[j] = (j >= lo && j < hi) ? sr[j] : __float_as_uint(NEG_INF);
        }
        float mx[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float acc = __uint_as_float(sr[32 * q4]);
#pragma unroll
          for (int j = 1; j < 31; j += 2)
            acc = fmax3f(acc, __uint_as_float(sr[32 * q4 + j]), __uint_as_float(sr[32 * q4 + j + 1]));
          mx[q4] = fmaxf(acc, __uint_as_float(sr[32 * q4 + 31]));
        }
        const float mt = fmax3f(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * sl2;
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + 8.0f;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m - m_new);
          l *= alpha;
          m = m_new;
        }
        const float mu = (m == NEG_INF) ? 0.f : m;
        const bool rescale = has_pv && __any_sync(0xffffffffu, need);
        const uint64_t sc2 = f2_pack(sl2, sl2);
        const uint64_t nm2 = f2_pack(-mu, -mu);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c2 = 64 * hh + 2 * j;
            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[c2]), __uint_as_float(sr[c2 + 1])),
                                       sc2, nm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            sum2[j & 3] = f2_add(sum2[j & 3], f2_pack(p0, p1));
            pk[j] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + 64 + 32 * hh, pk);
          if (hh == 0 && rescale) {
            uint32_t rr[32];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              tmem_ld32_sync(tO + 32 * ch, rr);
#pragma unroll
              for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * alpha);
              tmem_st32(tO + 32 * ch, rr);
            }
          }
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(f2_add(sum2[0], sum2[1]), a0, a1);
          f2_unpack(f2_add(sum2[2], sum2[3]), b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_remote(p_full);
        has_pv = 1;
      }
      if (!ok) break;
      // ---------------- epilogue: O = acc / l, LSE = ln 2 * (m + log2 l)
      if (!mbar_wait_bounded(bar(B_O_FULL + wg), unit_cnt & 1, tmo, a.err, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const bool live = l > 0.f;
      const float inv = live ? 1.f / l : 0.f;
      const float lse_v = live ? (m + lg2_approx(l)) * 0.69314718055994531f : NEG_INF;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rr[32];
        if (has_pv) {
          tmem_ld32_sync(tO + 32 * ch, rr);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) rr[j] = 0u;
        }
        if (valid) {
          if (OUT_FP32) {
            float* dst = static_cast<float*>(a.o) +
                         (static_cast<size_t>(t - a.row_base) * a.Hq + h) * D + 32 * ch;
            if (o_a32) {
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(rr[j + e]) * inv);
                st_global_v8(dst + j, w);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                float4 v4 = make_float4(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv,
                                        __uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
                *reinterpret_cast<float4*>(dst + j) = v4;
              }
            }
          } else {
            uint16_t* dst = static_cast<uint16_t*>(a.o) +
                            (static_cast<size_t>(t) * a.Hq + h) * D + 32 * ch;
            if (o_a32) {
#pragma unroll
              for (int j = 0; j < 32; j += 16) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  w[e] = pack_bf16x2(__uint_as_float(rr[j + 2 * e]) * inv, __uint_as_float(rr[j + 2 * e + 1]) * inv);
                st_global_v8(dst + j, w);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv);
                w.y = pack_bf16x2(__uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
                w.z = pack_bf16x2(__uint_as_float(rr[j + 4]) * inv, __uint_as_float(rr[j + 5]) * inv);
                w.w = pack_bf16x2(__uint_as_float(rr[j + 6]) * inv, __uint_as_float(rr[j + 7]) * inv);
                *reinterpret_cast<uint4*>(dst + j) = w;
              }
            }
          }
        }
      }
      if (valid) {
        if (OUT_FP32)
          a.lse[static_cast<size_t>(h) * a.n_rows + (t - a.row_base)] = lse_v;
        else
          a.lse[static_cast<size_t>(h) * a.T + t] = lse_v;
      }
      tc_fence_before();
    }
  }

  // Neither CTA leaves (or frees tensor memory) while the other may still
  // reach into its shared memory or while MMAs of the pair are in flight: the
  // first CTA's MMA lane has drained them before arriving here.
  tc_fence_before();
  __syncwarp();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

template <int OUT_FP32>
cudaError_t launch_pair(const AttnArgs& a, const void* tq, const void* tk, const void* tv, int n_pairs_hint,
                        cudaStream_t st) {
  using C = PCfg;
  auto kern = attn_tc_pair_kernel<OUT_FP32>;
  // Per-device set-up (the shared-memory attribute is a per-device setting,
  // and the cluster occupancy is queried once per device), shared by host
  // threads under a lock.
  static std::mutex mu;
  static bool configured[MAX_DEVICES] = {};
  static int max_clusters[MAX_DEVICES] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(384, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
      if (e != cudaSuccess) return e;
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
      max_clusters[dev] = n;
      configured[dev] = true;
    }
    clusters = max_clusters[dev];
  }
  if (n_pairs_hint > 0 && n_pairs_hint < clusters) clusters = n_pairs_hint;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  CUtensorMap mq, mk, mv;
  memcpy(&mq, tq, sizeof mq);
  memcpy(&mk, tk, sizeof mk);
  memcpy(&mv, tv, sizeof mv);
  return cudaLaunchKernelEx(&cfg, kern, a, mq, mk, mv);
}

}  // namespace

cudaError_t launch_attn_tc_pair(const AttnArgs& a, const void* tq, const void* tk64, const void* tv,
                                int n_pairs_hint, cudaStream_t st) {
  if (a.d != 128 || (a.Hq / a.Hkv) % 2 != 0) return cudaErrorInvalidValue;
  return a.out_mode ? launch_pair<1>(a, tq, tk64, tv, n_pairs_hint, st)
                    : launch_pair<0>(a, tq, tk64, tv, n_pairs_hint, st);
}

}  // namespace sp
