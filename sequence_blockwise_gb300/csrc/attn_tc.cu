// Blockwise packed attention on the 5th-generation tensor cores (sm_103a).
//
// One persistent CTA per SM walks work units (group, 256 query rows, query
// head). For each unit it visits the group's items in schedule order and each
// item's keys in 128-key tiles; every tile is one "partial attention" step
// (HSAP abstract) whose partial (O, LSE) is merged on chip into the running
// state by the log-sum-exp rule, the merge Ring Attention applies between
// ring steps (TASP abstract). Masks: same document, and key <= query when
// causal (HSAP abstract: no cross-contamination of packed documents).
//
// Roles (12 warps):
//   warp 0      TMA producer: Q tiles once per unit, K tiles into a 2-stage and
//               V tiles into a 3-stage ring (128-byte swizzled, as the MMA
//               reads them); it walks the tiles and publishes one record per K
//               stage (tile classes, last-of-unit).
//   warp 1      allocates tensor memory; lane 0 issues every tcgen05.mma.
//   warps 4-7   softmax for Q tile 0 (rows 0-127 of the unit).
//   warps 8-11  softmax for Q tile 1 (rows 128-255).
// Tensor memory (512 columns): S_i at column 128*i (fp32 128x128), the bf16
// probabilities P_i written back over columns [64,128) of S_i, and the output
// accumulators O_i at 256 + D*i.
// Per KV tile j the MMA order is QK0(j), PV1(j-1), QK1(j), PV0(j): each
// softmax warpgroup has two tensor-core steps of slack, and because MMAs from
// one thread execute in order, the completion of QK_i(j) also implies that
// PV_i(j-1) is done, so the softmax may rescale O_i without another wait.
// The running maximum is only moved when it grows by more than 2^8, so O is
// rarely rescaled (values stay <= 256 before normalisation).
// Tiles are classified per Q tile from the document bounds of its rows:
// SKIP (no valid pair: no load, no MMA), FULL (no mask), MASKED (per-row
// interval mask).

#include <cuda.h>

#include <mutex>

#include "sp_device.cuh"
#include "sp_tiles.cuh"

namespace sp {
namespace {

// Tile record the producer publishes with each K stage, so that the MMA lane
// does no tile bookkeeping of its own: bits [0,2) class of Q tile 0, [2,4)
// class of Q tile 1, REC_TILE when K/V were loaded, REC_LAST on the unit's last
// record (a unit without tiles publishes one record with REC_LAST only).
constexpr int REC_TILE = 16, REC_LAST = 32;

template <int D>
struct Cfg {
  // K is consumed by the first MMA of a tile and V by the last, so V buffers
  // are held longer: the V ring is one stage deeper than the K ring.
  static constexpr int KSTAGE = 2;
  static constexpr int VSTAGE = 3;
  static constexpr int KSUB = D / 64;             // 128-byte sub-tiles along d
  static constexpr int SUB_BYTES = 128 * 128;     // [128 rows][64 bf16]
  static constexpr int TILE_BYTES = KSUB * SUB_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGE * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + VSTAGE * TILE_BYTES;
  static constexpr int N_BARS = 20;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;   // TMEM address, abort flag
  static constexpr int OFF_REC = OFF_MISC + 8;             // one tile record per K stage
  static constexpr int OFF_URING = OFF_REC + 4 * KSTAGE;   // two unit ids in flight
  static constexpr int SMEM_ALLOC = OFF_URING + 8 + 1024;
  static constexpr int TM_S = 0;
  static constexpr int TM_O = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 0, 1);
};

// Barrier slots. KV_FULL[s] completes when both the K tile of K stage s and
// the V tile loaded with it have landed (one wait per tile for the MMA lane).
enum {
  B_Q_FULL = 0, B_Q_EMPTY = 1, B_KV_FULL = 2, B_K_EMPTY = 4, B_V_EMPTY = 6,
  B_S_FULL = 9, B_P_FULL = 11, B_O_FULL = 13, B_DRAIN = 15, B_U_FULL = 16, B_U_EMPTY = 18
};

// Units reach the MMA lane and the softmax warps through a two-slot ring filled
// by the producer lane: one consumer arrival from the MMA lane and one per
// softmax warp frees a slot.
constexpr int UNIT_CONSUMERS = 9;

// Non-blocking barrier tests run by the MMA lane just before the last MMA of a
// group, while that group is still executing: the MMA queue is shallow, so a
// test or wait between groups would leave the tensor core idle.
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

// S = Q K^T for one Q tile: D/16 MMAs of 128x128x16. Descriptor bases are
// fixed; only the 14-bit start address field (16-byte units) advances.
template <int D>
__device__ __forceinline__ int mma_qk(uint32_t d_t, uint64_t a0, uint64_t b0, const Probe& pa,
                                      const Probe& pb) {
  using C = Cfg<D>;
  int res = 0;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    if (kk == D / 16 - 1) res = run_probes(pa, pb);
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::SUB_BYTES + (kk & 3) * 32) >> 4);
    tc_mma_ss(d_t, a0 + off, b0 + off, C::IDESC_QK, kk > 0 ? 1u : 0u);
  }
  return res;
}

// Half h of O += P V: keys 64h .. 64h+63 (K steps 4h .. 4h+3); P read from
// tensor memory, V from shared memory (MN-major).
template <int D>
__device__ __forceinline__ int mma_pv_half(uint32_t d_t, uint32_t a_t, uint64_t b0, int h, int acc,
                                           const Probe& pa, const Probe& pb) {
  using C = Cfg<D>;
  int res = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kk = 4 * h + q;
    if (q == 3) res = run_probes(pa, pb);
    tc_mma_ts(d_t, a_t + 8 * kk, b0 + static_cast<uint64_t>(kk * (2048 >> 4)), C::IDESC_PV,
              (acc || kk > 0) ? 1u : 0u);
  }
  return res;
}

template <int D, int OUT_FP32>
__global__ void __launch_bounds__(384, 1)
attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmq,
               const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
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

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_EMPTY), 1);
    for (int s = 0; s < C::KSTAGE; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::VSTAGE; ++s) mbar_init(bar(B_V_EMPTY + s), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_P_FULL + i), 4);   // P_i stored (and O_i rescaled)
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
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_units = n_units_of(a);
  const int G = a.Hq / a.Hkv;
  const unsigned long long tmo = a.timeout_ns;

  // Register split: the producer/MMA warpgroup needs few registers, the two
  // softmax warpgroups hold a 128-column row of S each. 128*136 + 256*184 equals
  // the 384*168 the block is launched with.
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
      int armed_q = 0;
      uint32_t par_q = 0;
      bool ok = true;
      // Work units: claimed from the dynamic queue (longest key walks first, so
      // the tail is made of small units) or strided over the CTAs.
      int k_static = 0;
      auto fetch = [&]() -> int {
        int v;
        if (a.work_counter) {
          v = atomicAdd(a.work_counter, 1);
        } else {
          v = static_cast<int>(blockIdx.x) + k_static * static_cast<int>(gridDim.x);
          ++k_static;
        }
        return v < n_units ? v : -1;
      };
      int uslot = 0;
      uint32_t uph = 0;
      int u_next = fetch();
      for (;; ++unit_cnt) {
        const int u = u_next;
        if (!mbar_wait_bounded(bar(B_U_EMPTY + uslot), uph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
        uring[uslot] = u;
        mbar_arrive(bar(B_U_FULL + uslot));
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (u < 0) break;
        u_next = fetch();
        const UnitInfo ui = unit_info(a, u);
        const QTile qt[2] = {make_qtile(a, ui, 0), make_qtile(a, ui, 1)};
        const int hk = ui.h / G;
        if (!mbar_wait_bounded(bar(B_Q_EMPTY), (unit_cnt & 1) ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(B_Q_FULL), 2 * C::TILE_BYTES);
        armed_q = 1;
        par_q = unit_cnt & 1;
        for (int i = 0; i < 2; ++i)
          for (int s = 0; s < C::KSUB; ++s)
            tma_load_3d(sQ + i * C::TILE_BYTES + s * C::SUB_BYTES, &tmq, bar(B_Q_FULL), 64 * s,
                        ui.h, ui.q0 + 128 * i);
        // The tile walk runs one tile ahead so that each record can say
        // whether it is the unit's last.
        Cursor cur = make_cursor(a, ui, qt, a.causal);
        int ka = 0, kb = 0, cls[2] = {0, 0};
        bool have = next_tile(a, cur, qt, ka, kb, cls);
        if (!have) {
          if (!mbar_wait_bounded(bar(B_K_EMPTY + kst), kph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
          rec[kst] = REC_LAST;
          mbar_arrive(bar(B_KV_FULL + kst));
          if (++kst == C::KSTAGE) { kst = 0; kph ^= 1; }
        }
        while (have) {
          int nka, nkb, ncls[2];
          const bool nxt = next_tile(a, cur, qt, nka, nkb, ncls);
          if (!mbar_wait_bounded(bar(B_K_EMPTY + kst), kph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
          if (!mbar_wait_bounded(bar(B_V_EMPTY + vst), vph ^ 1, tmo, a.err, abort_flag)) { ok = false; break; }
          rec[kst] = REC_TILE | cls[0] | (cls[1] << 2) | (nxt ? 0 : REC_LAST);
          const uint32_t full = bar(B_KV_FULL + kst);
          mbar_arrive_expect_tx(full, 2 * C::TILE_BYTES);
          armed_k[kst] = 1;
          par_k[kst] = kph;
          for (int s = 0; s < C::KSUB; ++s)
            tma_load_3d(sK + kst * C::TILE_BYTES + s * C::SUB_BYTES, &tmk, full, 64 * s, hk, ka);
          for (int s = 0; s < C::KSUB; ++s)
            tma_load_3d(sV + vst * C::TILE_BYTES + s * C::SUB_BYTES, &tmv, full, 64 * s, hk, ka);
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
        // Aborting: let every copy already issued land before the block exits.
        volatile int no_abort = 0;
        const unsigned long long drain = 50000000ull;
        if (armed_q) mbar_wait_bounded(bar(B_Q_FULL), par_q, drain, a.err, &no_abort);
        for (int s = 0; s < C::KSTAGE; ++s)
          if (armed_k[s]) mbar_wait_bounded(bar(B_KV_FULL + s), par_k[s], drain, a.err, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sQ + C::TILE_BYTES, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sV, C::SUB_BYTES, 1024);
      uint32_t unit_cnt = 0, pcnt0 = 0, pcnt1 = 0;
      int kst = 0, vst = 0;
      uint32_t kph = 0;
      bool ok = true;
      const Probe none{0u, 0u, 0};
      const uint32_t dS0 = tmem + C::TM_S, dS1 = tmem + C::TM_S + 128;
      const uint32_t dO0 = tmem + C::TM_O, dO1 = tmem + C::TM_O + D;
      const uint32_t aP0 = dS0 + 64, aP1 = dS1 + 64;
      const uint64_t kstep = C::TILE_BYTES >> 4;

      bool rdy_k = false;
      int uslot = 0;
      uint32_t uph = 0;
      for (;; ++unit_cnt) {
        if (!mbar_wait_bounded(bar(B_U_FULL + uslot), uph, tmo, a.err, abort_flag)) { ok = false; break; }
        const int u = uring[uslot];
        mbar_arrive(bar(B_U_EMPTY + uslot));
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (u < 0) break;
        if (!mbar_wait_bounded(bar(B_Q_FULL), unit_cnt & 1, tmo, a.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
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
            const uint64_t bV = dv0 + static_cast<uint64_t>(vst) * kstep;
            const uint64_t bVp = dv0 + static_cast<uint64_t>(prev_vs) * kstep;
            const Probe p1{bar(B_P_FULL + 1), pcnt1 & 1, pv1};
            const Probe p0{bar(B_P_FULL + 0), pcnt0 & 1, c0 != CLS_SKIP};
            const Probe pk{bar(B_KV_FULL + nkst), nkph, 1};
            int got1 = 0, got0 = 0;
            if (c0 != CLS_SKIP) {
              got1 = mma_qk<D>(dS0, dq0, bK, p1, none) & 1;
              tc_commit(bar(B_S_FULL + 0));
            }
            if (pv1) {
              if (!got1 && !mbar_wait_bounded(p1.bar, p1.par, tmo, a.err, abort_flag)) { ok = false; break; }
              tc_fence_after();
              mma_pv_half<D>(dO1, aP1, bVp, 0, has_pv1, none, none);
              got0 = mma_pv_half<D>(dO1, aP1, bVp, 1, 1, p0, none) & 1;
              ++pcnt1;
              has_pv1 = 1;
            }
            if (have_prev) tc_commit(bar(B_V_EMPTY + prev_vs));
            if (c1 != CLS_SKIP) {
              const int g = mma_qk<D>(dS1, dq1, bK, got0 ? none : p0, none);
              got0 |= g & 1;
              tc_commit(bar(B_S_FULL + 1));
            }
            tc_commit(bar(B_K_EMPTY + kst));
            if (c0 != CLS_SKIP) {
              if (!got0 && !mbar_wait_bounded(p0.bar, p0.par, tmo, a.err, abort_flag)) { ok = false; break; }
              tc_fence_after();
              mma_pv_half<D>(dO0, aP0, bV, 0, has_pv0, none, none);
              rdy_k = mma_pv_half<D>(dO0, aP0, bV, 1, 1, (r & REC_LAST) ? none : pk, none) & 1;
              ++pcnt0;
              has_pv0 = 1;
            }
            have_prev = 1;
            prev_vs = vst;
            prev_c1 = c1;
            if (++vst == C::VSTAGE) vst = 0;
          } else {
            tc_commit(bar(B_K_EMPTY + kst));  // nothing was loaded: hand the slot back
          }
          kst = nkst;
          kph = nkph;
          if (r & REC_LAST) break;
        }
        if (!ok) break;
        // O_0 is complete once the PV0 issued so far are: the softmax warps of Q
        // tile 0 may read it out while the last PV1 still waits for its P.
        tc_commit(bar(B_O_FULL + 0));
        if (have_prev) {
          if (prev_c1 != CLS_SKIP) {
            const uint64_t bVp = dv0 + static_cast<uint64_t>(prev_vs) * kstep;
            if (!mbar_wait_bounded(bar(B_P_FULL + 1), pcnt1 & 1, tmo, a.err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            mma_pv_half<D>(dO1, aP1, bVp, 0, has_pv1, none, none);
            mma_pv_half<D>(dO1, aP1, bVp, 1, 1, none, none);
            ++pcnt1;
          }
          tc_commit(bar(B_V_EMPTY + prev_vs));
        }
        tc_commit(bar(B_Q_EMPTY));
        tc_commit(bar(B_O_FULL + 1));
      }
      // Every MMA issued has completed before tensor memory is released.
      volatile int no_abort = 0;
      tc_commit(bar(B_DRAIN));
      mbar_wait_bounded(bar(B_DRAIN), 0, 50000000ull, a.err, &no_abort);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    const int wg = (warp - 4) >> 2;       // which Q tile
    const int wq = warp & 3;              // tensor-memory lane quarter
    const int r = wq * 32 + lane;         // row within the Q tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + 128 * wg;
    const uint32_t tO = tmem + lane_off + C::TM_O + D * wg;
    const float sl2 = a.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    uint32_t s_cnt = 0, unit_cnt = 0;
    bool ok = true;
    int uslot = 0;
    uint32_t uph = 0;
    for (;; ++unit_cnt) {
      if (!mbar_wait_bounded(bar(B_U_FULL + uslot), uph, tmo, a.err, abort_flag)) { ok = false; break; }
      const int u = uring[uslot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_U_EMPTY + uslot));
      if (++uslot == 2) { uslot = 0; uph ^= 1; }
      if (u < 0) break;
      const UnitInfo ui = unit_info(a, u);
      const QTile qt[2] = {make_qtile(a, ui, 0), make_qtile(a, ui, 1)};
      const QTile my = wg ? qt[1] : qt[0];
      const int t = ui.q0 + 128 * wg + r;
      const bool valid = (t >= my.qa) && (t < my.qb);
      int rds = 0, rde = 0;
      if (valid) {
        const int dd = doc_of(a.cu, a.ndocs, t);
        rds = __ldg(a.cu + dd);
        rde = __ldg(a.cu + dd + 1);
      }
      const int rcausal_end = a.causal ? t + 1 : 0x7fffffff;
      float m = NEG_INF, l = 0.f;
      int has_pv = 0;
      Cursor cur = make_cursor(a, ui, qt, a.causal);
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
        // Row maximum: four independent chains of 3-input max.
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
        // p = 2^(s * scale * log2 e - m): packed FMA, then MUFU ex2, packed
        // row-sum; bf16 pairs are written back over columns [64, 128) of S,
        // in two halves to keep fewer registers live.
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
            // O_i rescale (rare: the row maximum grew by more than 2^8); it
            // must be done before P_i V is allowed to start.
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
        if (lane == 0) mbar_arrive(bar(B_P_FULL + wg));
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
                         (static_cast<size_t>(t - a.row_base) * a.Hq + ui.h) * D + 32 * ch;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 v4 = make_float4(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv,
                                      __uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
              *reinterpret_cast<float4*>(dst + j) = v4;
            }
          } else {
            uint16_t* dst = static_cast<uint16_t*>(a.o) +
                            (static_cast<size_t>(t) * a.Hq + ui.h) * D + 32 * ch;
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
      if (valid) {
        if (OUT_FP32)
          a.lse[static_cast<size_t>(ui.h) * a.n_rows + (t - a.row_base)] = lse_v;
        else
          a.lse[static_cast<size_t>(ui.h) * a.T + t] = lse_v;
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int OUT_FP32>
cudaError_t launch_one(const AttnArgs& a, const void* tq, const void* tk, const void* tv, int grid,
                       cudaStream_t st) {
  using C = Cfg<D>;
  auto kern = attn_tc_kernel<D, OUT_FP32>;
  // The shared-memory attribute is a per-device setting: set once per device,
  // under a lock shared by host threads.
  static std::mutex mu;
  static bool configured[MAX_DEVICES] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  CUtensorMap mq, mk, mv;
  memcpy(&mq, tq, sizeof mq);
  memcpy(&mk, tk, sizeof mk);
  memcpy(&mv, tv, sizeof mv);
  kern<<<grid, 384, C::SMEM_ALLOC, st>>>(a, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs& a, const void* tq, const void* tk, const void* tv,
                           int grid, cudaStream_t st) {
  if (a.d == 128) return a.out_mode ? launch_one<128, 1>(a, tq, tk, tv, grid, st)
                                    : launch_one<128, 0>(a, tq, tk, tv, grid, st);
  return a.out_mode ? launch_one<64, 1>(a, tq, tk, tv, grid, st)
                    : launch_one<64, 0>(a, tq, tk, tv, grid, st);
}

}  // namespace sp
