// Backward of the packed blockwise attention on the 5th-generation tensor
// cores (sm_103a): dQ, dK, dV from Q, K, V, O, dO and the forward's LSE.
//
// With P_ij = exp(scale q_i.k_j - LSE_i) over the valid keys of query i,
//   D_i = dO_i . O_i,  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j,
// dK and dV of a key/value head summing over the query heads of its group.
// Training with the sequence-parallel schedules runs this backward over the
// same chunk pairs (HSAP abstract: training throughput, tokens per GPU per
// second; TASP abstract: Ring Attention and its decompositions).
//
// Three kernels, launched in order on one stream:
//   bwd_rowdot   D_i per (row, head) into the workspace.
//   bwd_dkdv     one unit per (128-key tile, key/value head): K and V stay in
//                shared memory while every Q tile that can attend the keys is
//                streamed through (all query heads of the group). With keys on
//                the tensor-memory lanes: S^T = K Q^T and dP^T = V dO^T, the
//                compute warpgroup forms P^T and dS^T (scale folded in) in
//                place, then dV += P^T dO and dK += dS^T Q read their A operand
//                from tensor memory. TMEM: S^T, dP^T, dV, dK (128 columns each
//                for d = 128).
//   bwd_dq       one unit per (128-row Q tile, query head), walking the same
//                schedule items as the forward: S = Q K^T, dP = dO V^T, dS
//                written over S, dQ += dS K. TMEM: S, dP, dQ.
// Each kernel: warp 0 TMA producer, warp 1 TMEM owner and MMA lane, warps 4-7
// compute (one TMEM lane, i.e. one key or query row, per thread).

#include <cuda.h>

#include <cstring>

#include "sp_device.cuh"
#include "sp_tiles.cuh"

namespace sp {
namespace {

constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int KSUB = D / 64;
  static constexpr int SUB_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = KSUB * SUB_BYTES;
  static constexpr uint32_t IDESC_SS = idesc_bf16_f32(128, 128, 0, 0);  // both K-major
  static constexpr uint32_t IDESC_TS = idesc_bf16_f32(128, D, 0, 1);    // B MN-major
  static constexpr int TMEM_COLS = 512;
};

// Descriptor of a [128 rows][D] bf16 tile as a K-major operand (rows = M or N).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr) { return smem_desc_sw128(addr, 16, 1024); }
// The same tile as an MN-major B operand (rows = K, d = N).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t addr) {
  return smem_desc_sw128(addr, 128 * 128, 1024);
}

// D/16 MMAs of 128x128x16 contracting over d: C = A B^T with A, B K-major tiles.
template <int D>
__device__ __forceinline__ void mma_over_d(uint32_t d_t, uint64_t a0, uint64_t b0) {
  using C = BCfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::SUB_BYTES + (kk & 3) * 32) >> 4);
    tc_mma_ss(d_t, a0 + off, b0 + off, C::IDESC_SS, kk > 0 ? 1u : 0u);
  }
}

// 8 MMAs of 128xDx16 contracting over 128 rows: C (+)= A(tmem, bf16 pairs) B(MN-major).
template <int D>
__device__ __forceinline__ void mma_over_rows(uint32_t d_t, uint32_t a_t, uint64_t b0, int acc) {
  using C = BCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    tc_mma_ts(d_t, a_t + 8 * kk, b0 + static_cast<uint64_t>(kk * (2048 >> 4)), C::IDESC_TS,
              (acc || kk > 0) ? 1u : 0u);
}

// Writes 32 fp32 accumulator columns of one row as bf16.
__device__ __forceinline__ void store_row32_bf16(uint16_t* dst, const uint32_t (&rr)[32]) {
#pragma unroll
  for (int j = 0; j < 32; j += 8) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1]));
    w.y = pack_bf16x2(__uint_as_float(rr[j + 2]), __uint_as_float(rr[j + 3]));
    w.z = pack_bf16x2(__uint_as_float(rr[j + 4]), __uint_as_float(rr[j + 5]));
    w.w = pack_bf16x2(__uint_as_float(rr[j + 6]), __uint_as_float(rr[j + 7]));
    *reinterpret_cast<uint4*>(dst + j) = w;
  }
}

__device__ __forceinline__ void store_zero_row_bf16(uint16_t* dst, int n) {
  for (int j = 0; j < n; j += 8) *reinterpret_cast<uint4*>(dst + j) = make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------------ D_i

// D[h][t] = dO[t][h][:] . O[t][h][:] in fp32 from bf16; one warp per (t, h).
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ dout,
                                                         float* __restrict__ dvec, int T, int Hq,
                                                         int d) {
  const int lane = threadIdx.x & 31;
  const long long n = static_cast<long long>(T) * Hq;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       w < n; w += wstride) {
    const int t = static_cast<int>(w / Hq), h = static_cast<int>(w % Hq);
    const uint16_t* po = o + static_cast<size_t>(w) * d;
    const uint16_t* pd = dout + static_cast<size_t>(w) * d;
    float acc = 0.f;
    for (int c = 2 * lane; c < d; c += 64) {
      const uint32_t a = *reinterpret_cast<const uint32_t*>(po + c);
      const uint32_t b = *reinterpret_cast<const uint32_t*>(pd + c);
      acc = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), acc);
      acc = fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dvec[static_cast<size_t>(h) * T + t] = acc;
  }
}

// ------------------------------------------------------------------ dK, dV

template <int D>
struct KVCfg : BCfg<D> {
  using B = BCfg<D>;
  static constexpr int QSTAGE = 2;
  static constexpr int STAGE_BYTES = 2 * B::TILE_BYTES + 1024;  // Q, dO, LSE2[128], D[128]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = B::TILE_BYTES;
  static constexpr int OFF_QD = 2 * B::TILE_BYTES;
  static constexpr int OFF_BAR = OFF_QD + QSTAGE * STAGE_BYTES;
  static constexpr int N_BARS = 10;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
};

enum { KB_KV_FULL = 0, KB_KV_EMPTY = 1, KB_QD_FULL = 2, KB_QD_EMPTY = 4, KB_S_FULL = 6,
       KB_P_FULL = 7, KB_ACC_FULL = 8, KB_DRAIN = 9 };

struct KVUnit {
  int k0, k1, hk;  // keys [k0, k1) of key/value head hk
  int qa, qb;      // queries that may attend them
  int n_qt;        // Q tiles of 128 rows in [qa, qb)
};

__device__ __forceinline__ KVUnit kv_unit(const AttnArgs& a, int u) {
  KVUnit w;
  const int t = u / a.Hkv;
  w.hk = u - t * a.Hkv;
  w.k0 = 128 * t;
  w.k1 = min(w.k0 + 128, a.T);
  const int d0 = doc_of(a.cu, a.ndocs, w.k0);
  const int d1 = doc_of(a.cu, a.ndocs, w.k1 - 1);
  w.qa = a.causal ? w.k0 : __ldg(a.cu + d0);
  w.qb = __ldg(a.cu + d1 + 1);
  w.n_qt = (w.qb - w.qa + 127) / 128;
  return w;
}

template <int D>
__global__ void __launch_bounds__(256, 1)
bwd_dkdv_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const __grid_constant__ CUtensorMap tmdo) {
  using C = KVCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sQD = sbase + C::OFF_QD;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnArgs& f = a.fwd;

  if (threadIdx.x == 0) {
    mbar_init(bar(KB_KV_FULL), 1);
    mbar_init(bar(KB_KV_EMPTY), 1);
    for (int s = 0; s < C::QSTAGE; ++s) {
      mbar_init(bar(KB_QD_FULL + s), 32);  // every producer lane stores LSE/D; lane 0 arms the bytes
      mbar_init(bar(KB_QD_EMPTY + s), 1);
    }
    mbar_init(bar(KB_S_FULL), 1);
    mbar_init(bar(KB_P_FULL), 4);
    mbar_init(bar(KB_ACC_FULL), 1);
    mbar_init(bar(KB_DRAIN), 1);
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
  const int G = f.Hq / f.Hkv;
  const int n_units = ((f.T + 127) / 128) * f.Hkv;
  const unsigned long long tmo = f.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t unit_cnt = 0, qph = 0;
    int qst = 0;
    int armed_kv = 0, armed_qd[C::QSTAGE] = {0, 0};
    uint32_t par_kv = 0, par_qd[C::QSTAGE] = {0, 0};
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
      const KVUnit w = kv_unit(f, u);
      bool got = true;
      if (lane == 0) {
        got = mbar_wait_bounded(bar(KB_KV_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag);
        if (got) {
          mbar_arrive_expect_tx(bar(KB_KV_FULL), 2 * C::TILE_BYTES);
          armed_kv = 1;
          par_kv = unit_cnt & 1;
          for (int s = 0; s < C::KSUB; ++s) {
            tma_load_3d(sK + s * C::SUB_BYTES, &tmk, bar(KB_KV_FULL), 64 * s, w.hk, w.k0);
            tma_load_3d(sV + s * C::SUB_BYTES, &tmv, bar(KB_KV_FULL), 64 * s, w.hk, w.k0);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) { ok = false; break; }
      for (int step = 0; step < w.n_qt * G; ++step) {
        const int h = w.hk * G + step % G;
        const int q0 = w.qa + 128 * (step / G);
        const bool e = mbar_wait_bounded(bar(KB_QD_EMPTY + qst), qph ^ 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        float* lse2 = reinterpret_cast<float*>(smem + C::OFF_QD + qst * C::STAGE_BYTES + 2 * C::TILE_BYTES);
        float* dd = lse2 + 128;
        for (int idx = lane; idx < 128; idx += 32) {
          const int row = q0 + idx;
          const bool in = row < w.qb;
          lse2[idx] = in ? __ldg(a.lse + static_cast<size_t>(h) * f.T + row) * LOG2E : 0.f;
          dd[idx] = in ? __ldg(a.dvec + static_cast<size_t>(h) * f.T + row) : 0.f;
        }
        const uint32_t full = bar(KB_QD_FULL + qst);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, 2 * C::TILE_BYTES);
          const uint32_t sq = sQD + qst * C::STAGE_BYTES;
          for (int s = 0; s < C::KSUB; ++s) {
            tma_load_3d(sq + s * C::SUB_BYTES, &tmq, full, 64 * s, h, q0);
            tma_load_3d(sq + C::TILE_BYTES + s * C::SUB_BYTES, &tmdo, full, 64 * s, h, q0);
          }
          armed_qd[qst] = 1;
          par_qd[qst] = qph;
        } else {
          mbar_arrive(full);
        }
        if (++qst == C::QSTAGE) { qst = 0; qph ^= 1; }
      }
    }
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      if (armed_kv) mbar_wait_bounded(bar(KB_KV_FULL), par_kv, 50000000ull, f.err, &no_abort);
      for (int s = 0; s < C::QSTAGE; ++s)
        if (armed_qd[s]) mbar_wait_bounded(bar(KB_QD_FULL + s), par_qd[s], 50000000ull, f.err, &no_abort);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA lane
    if (lane == 0) {
      const uint64_t dKa = desc_kmajor(sK), dVa = desc_kmajor(sV);
      const uint32_t tS = tmem + C::TM_S, tdP = tmem + C::TM_DP;
      const uint32_t tdV = tmem + C::TM_DV, tdK = tmem + C::TM_DK;
      uint32_t unit_cnt = 0, qph = 0, pcnt = 0;
      int qst = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
        const KVUnit w = kv_unit(f, u);
        if (!mbar_wait_bounded(bar(KB_KV_FULL), unit_cnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        int has_acc = 0;
        for (int step = 0; step < w.n_qt * G; ++step) {
          if (!mbar_wait_bounded(bar(KB_QD_FULL + qst), qph, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sq = sQD + qst * C::STAGE_BYTES, sdo = sq + C::TILE_BYTES;
          mma_over_d<D>(tS, dKa, desc_kmajor(sq));    // S^T = K Q^T
          mma_over_d<D>(tdP, dVa, desc_kmajor(sdo));  // dP^T = V dO^T
          tc_commit(bar(KB_S_FULL));
          if (!mbar_wait_bounded(bar(KB_P_FULL), pcnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
          ++pcnt;
          tc_fence_after();
          mma_over_rows<D>(tdV, tS, desc_mnmajor(sdo), has_acc);  // dV += P^T dO
          mma_over_rows<D>(tdK, tdP, desc_mnmajor(sq), has_acc);  // dK += dS^T Q
          tc_commit(bar(KB_QD_EMPTY + qst));
          has_acc = 1;
          if (++qst == C::QSTAGE) { qst = 0; qph ^= 1; }
        }
        if (!ok) break;
        tc_commit(bar(KB_KV_EMPTY));
        tc_commit(bar(KB_ACC_FULL));
      }
      volatile int no_abort = 0;
      tc_commit(bar(KB_DRAIN));
      mbar_wait_bounded(bar(KB_DRAIN), 0, 50000000ull, f.err, &no_abort);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S, tdP = tmem + lane_off + C::TM_DP;
    const uint32_t tdV = tmem + lane_off + C::TM_DV, tdK = tmem + lane_off + C::TM_DK;
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, scnt = 0, qph = 0;
    int qst = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
      const KVUnit w = kv_unit(f, u);
      const int j = w.k0 + r;
      const bool kvalid = j < w.k1;
      int lo = 0, hi = 0;  // queries that may attend key j
      if (kvalid) {
        const int dj = doc_of(f.cu, f.ndocs, j);
        lo = f.causal ? j : __ldg(f.cu + dj);
        hi = min(__ldg(f.cu + dj + 1), w.qb);
      }
      int has_acc = 0;
      for (int step = 0; step < w.n_qt * G; ++step) {
        const int q0 = w.qa + 128 * (step / G);
        bool e = mbar_wait_bounded(bar(KB_S_FULL), scnt & 1, tmo, f.err, abort_flag);
        e = e && mbar_wait_bounded(bar(KB_QD_FULL + qst), qph, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        ++scnt;
        tc_fence_after();
        const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_QD + qst * C::STAGE_BYTES + 2 * C::TILE_BYTES);
        const float* dd = lse2 + 128;
        const int clo = kvalid ? max(lo, q0) - q0 : 0;
        const int chi = kvalid ? min(hi, q0 + 128) - q0 : 0;
        uint32_t x[128];  // S^T of this key row, then P^T in place (fp32 bits)
        tmem_ld128_sync(tS, x);
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const int cc = c + e4;
            const float pv = ex2_approx(fmaf(__uint_as_float(x[cc]), sl2, -lv[e4]));
            x[cc] = __float_as_uint((cc >= clo && cc < chi) ? pv : 0.f);
          }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(x[64 * hh + 2 * c]), __uint_as_float(x[64 * hh + 2 * c + 1]));
          tmem_st32(tS + 32 * hh, pk);  // P^T, queries 64 hh .. 64 hh + 63
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t dp[32];
          tmem_ld32_sync(tdP + 32 * ch, dp);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int q = 32 * ch + c;
            const float2 d2 = *reinterpret_cast<const float2*>(dd + q);
            const float s0 = __uint_as_float(x[q]) * (__uint_as_float(dp[c]) - d2.x) * scale;
            const float s1 = __uint_as_float(x[q + 1]) * (__uint_as_float(dp[c + 1]) - d2.y) * scale;
            pk[c >> 1] = pack_bf16x2(s0, s1);
          }
          tmem_st16(tdP + 16 * ch, pk);  // dS^T with the scale folded in
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_P_FULL));
        has_acc = 1;
        if (++qst == C::QSTAGE) { qst = 0; qph ^= 1; }
      }
      if (!ok) break;
      const bool e = mbar_wait_bounded(bar(KB_ACC_FULL), unit_cnt & 1, tmo, f.err, abort_flag);
      if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rv[32], rk[32];
        if (has_acc) {
          tmem_ld32_sync(tdV + 32 * ch, rv);
          tmem_ld32_sync(tdK + 32 * ch, rk);
        }
        if (kvalid) {
          const size_t off = (static_cast<size_t>(j) * f.Hkv + w.hk) * D + 32 * ch;
          if (has_acc) {
            store_row32_bf16(static_cast<uint16_t*>(a.dv) + off, rv);
            store_row32_bf16(static_cast<uint16_t*>(a.dk) + off, rk);
          } else {
            store_zero_row_bf16(static_cast<uint16_t*>(a.dv) + off, 32);
            store_zero_row_bf16(static_cast<uint16_t*>(a.dk) + off, 32);
          }
        }
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

// ------------------------------------------------------------------ dQ

template <int D>
struct QCfg : BCfg<D> {
  using B = BCfg<D>;
  static constexpr int KSTAGE = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = B::TILE_BYTES;
  static constexpr int OFF_K = 2 * B::TILE_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGE * B::TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + KSTAGE * B::TILE_BYTES;
  static constexpr int N_BARS = 12;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DQ = 256;
};

enum { QB_Q_FULL = 0, QB_Q_EMPTY = 1, QB_KV_FULL = 2, QB_KV_EMPTY = 4, QB_S_FULL = 6, QB_P_FULL = 7,
       QB_ACC_FULL = 8, QB_DRAIN = 9 };

template <int D>
__global__ void __launch_bounds__(256, 1)
bwd_dq_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tmq,
              const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
              const __grid_constant__ CUtensorMap tmdo) {
  using C = QCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO, sK = sbase + C::OFF_K,
                 sV = sbase + C::OFF_V;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(QB_Q_FULL), 1);
    mbar_init(bar(QB_Q_EMPTY), 1);
    for (int s = 0; s < C::KSTAGE; ++s) {
      mbar_init(bar(QB_KV_FULL + s), 1);
      mbar_init(bar(QB_KV_EMPTY + s), 1);
    }
    mbar_init(bar(QB_S_FULL), 1);
    mbar_init(bar(QB_P_FULL), 4);
    mbar_init(bar(QB_ACC_FULL), 1);
    mbar_init(bar(QB_DRAIN), 1);
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
  const AttnArgs& f = a.fwd;
  const int n_units = n_units_of(f);
  const int G = f.Hq / f.Hkv;
  const unsigned long long tmo = f.timeout_ns;

  // The unit's single Q tile; the second slot of the shared tile walk stays empty.
  auto unit_tiles = [&](const UnitInfo& ui, QTile (&qt)[2]) {
    qt[0] = make_qtile(f, ui, 0);
    qt[1].qa = qt[1].qb = qt[1].ds = qt[1].de = qt[1].one_doc = 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kv_cnt = 0, unit_cnt = 0;
      int armed_q = 0, armed_kv[C::KSTAGE] = {0, 0};
      uint32_t par_q = 0, par_kv[C::KSTAGE] = {0, 0};
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
        const UnitInfo ui = unit_info(f, u);
        QTile qt[2];
        unit_tiles(ui, qt);
        const int hk = ui.h / G;
        if (!mbar_wait_bounded(bar(QB_Q_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(QB_Q_FULL), 2 * C::TILE_BYTES);
        armed_q = 1;
        par_q = unit_cnt & 1;
        for (int s = 0; s < C::KSUB; ++s) {
          tma_load_3d(sQ + s * C::SUB_BYTES, &tmq, bar(QB_Q_FULL), 64 * s, ui.h, ui.q0);
          tma_load_3d(sDO + s * C::SUB_BYTES, &tmdo, bar(QB_Q_FULL), 64 * s, ui.h, ui.q0);
        }
        Cursor cur = make_cursor(ui, qt, f.causal);
        int ka, kb, cls[2];
        while (next_tile(f, cur, qt, ka, kb, cls)) {
          const int st = kv_cnt % C::KSTAGE;
          const uint32_t ph = (kv_cnt / C::KSTAGE) & 1;
          if (!mbar_wait_bounded(bar(QB_KV_EMPTY + st), ph ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(QB_KV_FULL + st), 2 * C::TILE_BYTES);
          armed_kv[st] = 1;
          par_kv[st] = ph;
          for (int s = 0; s < C::KSUB; ++s) {
            tma_load_3d(sK + st * C::TILE_BYTES + s * C::SUB_BYTES, &tmk, bar(QB_KV_FULL + st), 64 * s, hk, ka);
            tma_load_3d(sV + st * C::TILE_BYTES + s * C::SUB_BYTES, &tmv, bar(QB_KV_FULL + st), 64 * s, hk, ka);
          }
          ++kv_cnt;
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        if (armed_q) mbar_wait_bounded(bar(QB_Q_FULL), par_q, 50000000ull, f.err, &no_abort);
        for (int s = 0; s < C::KSTAGE; ++s)
          if (armed_kv[s]) mbar_wait_bounded(bar(QB_KV_FULL + s), par_kv[s], 50000000ull, f.err, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA lane
    if (lane == 0) {
      const uint64_t dQa = desc_kmajor(sQ), dDOa = desc_kmajor(sDO);
      const uint32_t tS = tmem + C::TM_S, tdP = tmem + C::TM_DP, tdQ = tmem + C::TM_DQ;
      uint32_t kv_cnt = 0, unit_cnt = 0, pcnt = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
        const UnitInfo ui = unit_info(f, u);
        QTile qt[2];
        unit_tiles(ui, qt);
        if (!mbar_wait_bounded(bar(QB_Q_FULL), unit_cnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        int has_acc = 0;
        Cursor cur = make_cursor(ui, qt, f.causal);
        int ka, kb, cls[2];
        while (next_tile(f, cur, qt, ka, kb, cls)) {
          const int st = kv_cnt % C::KSTAGE;
          const uint32_t ph = (kv_cnt / C::KSTAGE) & 1;
          if (!mbar_wait_bounded(bar(QB_KV_FULL + st), ph, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sk = sK + st * C::TILE_BYTES, sv = sV + st * C::TILE_BYTES;
          mma_over_d<D>(tS, dQa, desc_kmajor(sk));    // S = Q K^T
          mma_over_d<D>(tdP, dDOa, desc_kmajor(sv));  // dP = dO V^T
          tc_commit(bar(QB_S_FULL));
          if (!mbar_wait_bounded(bar(QB_P_FULL), pcnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
          ++pcnt;
          tc_fence_after();
          mma_over_rows<D>(tdQ, tS, desc_mnmajor(sk), has_acc);  // dQ += dS K
          tc_commit(bar(QB_KV_EMPTY + st));
          has_acc = 1;
          ++kv_cnt;
        }
        if (!ok) break;
        tc_commit(bar(QB_Q_EMPTY));
        tc_commit(bar(QB_ACC_FULL));
      }
      volatile int no_abort = 0;
      tc_commit(bar(QB_DRAIN));
      mbar_wait_bounded(bar(QB_DRAIN), 0, 50000000ull, f.err, &no_abort);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S, tdP = tmem + lane_off + C::TM_DP;
    const uint32_t tdQ = tmem + lane_off + C::TM_DQ;
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, scnt = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
      const UnitInfo ui = unit_info(f, u);
      QTile qt[2];
      unit_tiles(ui, qt);
      const int t = ui.q0 + r;
      const bool valid = t >= qt[0].qa && t < qt[0].qb;
      int rds = 0, rde = 0;
      float lse2 = 0.f, di = 0.f;
      if (valid) {
        const int dd = doc_of(f.cu, f.ndocs, t);
        rds = __ldg(f.cu + dd);
        rde = __ldg(f.cu + dd + 1);
        lse2 = __ldg(a.lse + static_cast<size_t>(ui.h) * f.T + t) * LOG2E;
        di = __ldg(a.dvec + static_cast<size_t>(ui.h) * f.T + t);
      }
      const int rcausal_end = f.causal ? t + 1 : 0x7fffffff;
      int has_acc = 0;
      Cursor cur = make_cursor(ui, qt, f.causal);
      int ka, kb, cls[2];
      while (next_tile(f, cur, qt, ka, kb, cls)) {
        const bool e = mbar_wait_bounded(bar(QB_S_FULL), scnt & 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        ++scnt;
        tc_fence_after();
        int lo = 0, hi = 128;
        if (cls[0] == CLS_MASKED) {
          lo = valid ? max(ka, rds) - ka : 0;
          hi = valid ? min(min(kb, rde), rcausal_end) - ka : 0;
        }
        uint32_t x[128];  // S of this row, then P in place (fp32 bits)
        tmem_ld128_sync(tS, x);
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float pv = ex2_approx(fmaf(__uint_as_float(x[c]), sl2, -lse2));
          x[c] = __float_as_uint((c >= lo && c < hi) ? pv : 0.f);
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t dp[32];
          tmem_ld32_sync(tdP + 32 * ch, dp);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float d0 = __uint_as_float(x[32 * ch + c]) * (__uint_as_float(dp[c]) - di) * scale;
            const float d1 = __uint_as_float(x[32 * ch + c + 1]) * (__uint_as_float(dp[c + 1]) - di) * scale;
            pk[c >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tS + 16 * ch, pk);  // dS over the (already read) S columns
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_P_FULL));
        has_acc = 1;
      }
      if (!ok) break;
      const bool e = mbar_wait_bounded(bar(QB_ACC_FULL), unit_cnt & 1, tmo, f.err, abort_flag);
      if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rq[32];
        if (has_acc) tmem_ld32_sync(tdQ + 32 * ch, rq);
        if (valid) {
          uint16_t* dst = static_cast<uint16_t*>(a.dq) + (static_cast<size_t>(t) * f.Hq + ui.h) * D + 32 * ch;
          if (has_acc) store_row32_bf16(dst, rq);
          else store_zero_row_bf16(dst, 32);
        }
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

template <typename Cfg, typename K>
cudaError_t launch_cfg(K kern, int grid, cudaStream_t st, const BwdArgs& a, const CUtensorMap& q,
                       const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<grid, 256, Cfg::SMEM_ALLOC, st>>>(a, q, k, v, dout);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_rowdot(const void* o, const void* dout, float* dvec, int T, int Hq, int d,
                              int grid, cudaStream_t st) {
  bwd_rowdot_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(o),
                                         static_cast<const uint16_t*>(dout), dvec, T, Hq, d);
  return cudaGetLastError();
}

cudaError_t launch_bwd_tc(const BwdArgs& a, const void* tq, const void* tk, const void* tv,
                          const void* tdo, int grid, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo;
  memcpy(&mq, tq, sizeof mq);
  memcpy(&mk, tk, sizeof mk);
  memcpy(&mv, tv, sizeof mv);
  memcpy(&mdo, tdo, sizeof mdo);
  const long long kv_units = static_cast<long long>((a.fwd.T + 127) / 128) * a.fwd.Hkv;
  const int kv_grid = static_cast<int>(kv_units < grid ? kv_units : grid);
  cudaError_t e;
  if (a.fwd.d == 128) {
    e = launch_cfg<QCfg<128>>(bwd_dq_kernel<128>, grid, st, a, mq, mk, mv, mdo);
    if (e != cudaSuccess) return e;
    return launch_cfg<KVCfg<128>>(bwd_dkdv_kernel<128>, kv_grid, st, a, mq, mk, mv, mdo);
  }
  e = launch_cfg<QCfg<64>>(bwd_dq_kernel<64>, grid, st, a, mq, mk, mv, mdo);
  if (e != cudaSuccess) return e;
  return launch_cfg<KVCfg<64>>(bwd_dkdv_kernel<64>, kv_grid, st, a, mq, mk, mv, mdo);
}

}  // namespace sp
