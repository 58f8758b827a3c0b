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
//   bwd_dkdv     one unit per (key/value head, 128-key tile), head-major so
//                that the CTAs running at one time share the Q and dO of one
//                head group in L2. K and V stay in shared memory while every
//                64-row Q block that can attend the keys is streamed through
//                (all query heads of the group). Keys sit on the tensor-memory
//                lanes: S^T = K Q^T and dP^T = V dO^T (128 x 64 each, double
//                buffered), the compute warpgroup turns them into P^T and dS^T
//                (scale folded in) in place, then dV += P^T dO and
//                dK += dS^T Q read their A operand from tensor memory.
//   bwd_dq       one unit per (128-row Q tile, query head), walking the same
//                schedule items as the forward in 64-key steps: S = Q K^T and
//                dP = dO V^T (128 x 64, double buffered), dS written over S,
//                dQ += dS K.
// Double buffering lets the MMA lane issue step n+1's S and dP while step n
// is being worked on. Each kernel: warp 0 TMA producer, warp 1 TMEM owner and
// MMA lane, warps 4-7 and 8-11 two compute warpgroups that take alternate
// steps (step g uses buffer g & 1 and warpgroup g & 1; one TMEM lane, i.e.
// one key or query row, per thread) and split the epilogue. All tensor maps use {64 dims, 1 head, 64 rows}
// boxes with 128-byte swizzle; a 128-row tile is two boxes, row r at r x 128
// bytes of each 64-dim sub-tile, which is the same layout one 128-row box gives.

#include <cuda.h>

#include <cstring>

#include "sp_device.cuh"
#include "sp_tiles.cuh"

namespace sp {
namespace {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int NSTEP = 64;  // rows of the streamed operand per step

template <int D>
struct BCfg {
  static constexpr int KSUB = D / 64;                  // 64-dim sub-tiles
  static constexpr int SUB128 = 128 * 128;             // bytes of a 128-row sub-tile
  static constexpr int SUB64 = 64 * 128;               // bytes of a 64-row sub-tile
  static constexpr int TILE128 = KSUB * SUB128;
  static constexpr int TILE64 = KSUB * SUB64;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, NSTEP, 0, 0);  // both K-major
  static constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, D, 0, 1);    // B MN-major
  static constexpr int TMEM_COLS = 512;
};

// K-major operand descriptor (rows = M or N, 64 dims per 128-byte row).
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return smem_desc_sw128(addr, 16, 1024); }
// MN-major B operand over a tile of 64 rows (K) x D (N): the next 64 columns
// of N start one 64-row sub-tile further on.
__device__ __forceinline__ uint64_t desc_mn64(uint32_t addr) { return smem_desc_sw128(addr, 64 * 128, 1024); }

// D/16 MMAs contracting over d: C[128 x 64] = A[128 rows] B[64 rows]^T, both
// K-major; A is a 128-row tile, B a 64-row tile.
template <int D>
__device__ __forceinline__ void mma_s(uint32_t d_t, uint32_t a_addr, uint32_t b_addr) {
  using C = BCfg<D>;
  const uint64_t a0 = desc_k(a_addr), b0 = desc_k(b_addr);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t ao = static_cast<uint64_t>(((kk >> 2) * C::SUB128 + (kk & 3) * 32) >> 4);
    const uint64_t bo = static_cast<uint64_t>(((kk >> 2) * C::SUB64 + (kk & 3) * 32) >> 4);
    tc_mma_ss(d_t, a0 + ao, b0 + bo, C::IDESC_S, kk > 0 ? 1u : 0u);
  }
}

// 4 MMAs contracting over 64 rows: C[128 x D] (+)= A(tmem, 32 columns of bf16
// pairs) B(64 rows x D, MN-major).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t d_t, uint32_t a_t, uint32_t b_addr, int acc) {
  using C = BCfg<D>;
  const uint64_t b0 = desc_mn64(b_addr);
#pragma unroll
  for (int kk = 0; kk < NSTEP / 16; ++kk)
    tc_mma_ts(d_t, a_t + 8 * kk, b0 + static_cast<uint64_t>(kk * (2048 >> 4)), C::IDESC_ACC,
              (acc || kk > 0) ? 1u : 0u);
}

// TMA of a 64-row block (all D dims) of one head into a 64-row tile.
template <int D>
__device__ __forceinline__ void load_rows64(uint32_t dst, const CUtensorMap* m, uint32_t bar, int h,
                                            int row0) {
  using C = BCfg<D>;
#pragma unroll
  for (int s = 0; s < C::KSUB; ++s) tma_load_3d(dst + s * C::SUB64, m, bar, 64 * s, h, row0);
}

// TMA of a 128-row block as two 64-row boxes into a 128-row tile (row0 < T).
// When the second box would start at or past row T it is taken from row T-1
// instead, so that no box lies wholly outside the tensor; those tile rows
// belong to no valid token and every use of them is masked.
template <int D>
__device__ __forceinline__ void load_rows128(uint32_t dst, const CUtensorMap* m, uint32_t bar, int h,
                                             int row0, int T) {
  using C = BCfg<D>;
  const int row1 = row0 + 64 < T ? row0 + 64 : T - 1;
#pragma unroll
  for (int s = 0; s < C::KSUB; ++s) {
    tma_load_3d(dst + s * C::SUB128, m, bar, 64 * s, h, row0);
    tma_load_3d(dst + s * C::SUB128 + C::SUB64, m, bar, 64 * s, h, row1);
  }
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

// Softmax-gradient work of one step for one TMEM lane (one row of the
// 128-lane operand, 64 columns of the streamed operand): P from S, then dS
// from P and dP. lse2_of(c) / dd_of(c) give the log2-scaled LSE and D of
// column c's query (or the row's own when they are per row). Columns outside
// [lo, hi) get P = dS = 0. P is packed to bf16 pairs into the S columns
// (32 columns) when keep_p; dS (scale folded in) is packed into dst_ds.
template <bool kKeepP, typename LseF, typename DF>
__device__ __forceinline__ void grad_step(uint32_t t_s, uint32_t t_dp, uint32_t dst_ds, int lo, int hi,
                                          float sl2, float scale, LseF lse2_of, DF dd_of) {
  uint32_t x[64];
  {
    uint32_t a[32];
    tmem_ld32_sync(t_s, a);
#pragma unroll
    for (int c = 0; c < 32; ++c) x[c] = a[c];
    tmem_ld32_sync(t_s + 32, a);
#pragma unroll
    for (int c = 0; c < 32; ++c) x[32 + c] = a[c];
  }
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    const float pv = ex2_approx(fmaf(__uint_as_float(x[c]), sl2, -lse2_of(c)));
    x[c] = __float_as_uint((c >= lo && c < hi) ? pv : 0.f);
  }
  if (kKeepP) {
    uint32_t pk[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1]));
    tmem_st32(t_s, pk);
  }
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    uint32_t dp[32];
    tmem_ld32_sync(t_dp + 32 * ch, dp);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const int q = 32 * ch + c;
      const float s0 = __uint_as_float(x[q]) * (__uint_as_float(dp[c]) - dd_of(q)) * scale;
      const float s1 = __uint_as_float(x[q + 1]) * (__uint_as_float(dp[c + 1]) - dd_of(q + 1)) * scale;
      pk[c >> 1] = pack_bf16x2(s0, s1);
    }
    tmem_st16(dst_ds + 16 * ch, pk);
  }
  tmem_wait_st();
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
  static constexpr int QSTAGE = 4;
  static constexpr int STAGE_BYTES = 2 * B::TILE64 + 1024;  // Q, dO, LSE2[64], D[64]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = B::TILE128;
  static constexpr int OFF_QD = 2 * B::TILE128;
  static constexpr int OFF_BAR = OFF_QD + QSTAGE * STAGE_BYTES;
  static constexpr int N_BARS = 17;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
};

enum { KB_KV_FULL = 0, KB_KV_EMPTY = 1, KB_QD_FULL = 2, KB_QD_EMPTY = 6, KB_S_FULL = 10,
       KB_P_FULL = 12, KB_ACC_FULL = 14, KB_DRAIN = 15, KB_ACC_EMPTY = 16 };

struct KVUnit {
  int k0, k1, hk;  // keys [k0, k1) of key/value head hk
  int qa, qb;      // queries that may attend them
  int n_steps;     // 64-row Q blocks in [qa, qb) times the heads of the group
};

// Units are head-major: all key tiles of head 0, then head 1, ...
__device__ __forceinline__ KVUnit kv_unit(const AttnArgs& a, int u) {
  KVUnit w;
  const int n_tiles = (a.T + 127) / 128;
  w.hk = u / n_tiles;
  const int t = u - w.hk * n_tiles;
  w.k0 = 128 * t;
  w.k1 = min(w.k0 + 128, a.T);
  const int d0 = doc_of(a.cu, a.ndocs, w.k0);
  const int d1 = doc_of(a.cu, a.ndocs, w.k1 - 1);
  w.qa = a.causal ? w.k0 : __ldg(a.cu + d0);
  w.qb = __ldg(a.cu + d1 + 1);
  w.n_steps = ((w.qb - w.qa + NSTEP - 1) / NSTEP) * (a.Hq / a.Hkv);
  return w;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(KB_S_FULL + b), 1);
      mbar_init(bar(KB_P_FULL + b), 4);
    }
    mbar_init(bar(KB_ACC_FULL), 1);
    mbar_init(bar(KB_DRAIN), 1);
    mbar_init(bar(KB_ACC_EMPTY), 8);  // every compute warp, after its part of the epilogue
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
    uint32_t unit_cnt = 0, gs = 0;
    int armed_kv = 0, armed_qd[C::QSTAGE] = {0, 0, 0, 0};
    uint32_t par_kv = 0, par_qd[C::QSTAGE] = {0, 0, 0, 0};
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
      const KVUnit w = kv_unit(f, u);
      bool got = true;
      if (lane == 0) {
        got = mbar_wait_bounded(bar(KB_KV_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag);
        if (got) {
          mbar_arrive_expect_tx(bar(KB_KV_FULL), 2 * C::TILE128);
          armed_kv = 1;
          par_kv = unit_cnt & 1;
          load_rows128<D>(sK, &tmk, bar(KB_KV_FULL), w.hk, w.k0, f.T);
          load_rows128<D>(sV, &tmv, bar(KB_KV_FULL), w.hk, w.k0, f.T);
        }
      }
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) { ok = false; break; }
      for (int step = 0; step < w.n_steps; ++step, ++gs) {
        const int st = gs % C::QSTAGE;
        const uint32_t ph = (gs / C::QSTAGE) & 1;
        const int h = w.hk * G + step % G;
        const int q0 = w.qa + NSTEP * (step / G);
        const bool e = mbar_wait_bounded(bar(KB_QD_EMPTY + st), ph ^ 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        float* lse2 = reinterpret_cast<float*>(smem + C::OFF_QD + st * C::STAGE_BYTES + 2 * C::TILE64);
        float* dd = lse2 + NSTEP;
        for (int idx = lane; idx < NSTEP; idx += 32) {
          const int row = q0 + idx;
          const bool in = row < w.qb;
          lse2[idx] = in ? __ldg(a.lse + static_cast<size_t>(h) * f.T + row) * LOG2E : 0.f;
          dd[idx] = in ? __ldg(a.dvec + static_cast<size_t>(h) * f.T + row) : 0.f;
        }
        const uint32_t full = bar(KB_QD_FULL + st);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, 2 * C::TILE64);
          const uint32_t sq = sQD + st * C::STAGE_BYTES;
          load_rows64<D>(sq, &tmq, full, h, q0);
          load_rows64<D>(sq + C::TILE64, &tmdo, full, h, q0);
          armed_qd[st] = 1;
          par_qd[st] = ph;
        } else {
          mbar_arrive(full);
        }
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
      const uint32_t tdV = tmem + C::TM_DV, tdK = tmem + C::TM_DK;
      uint32_t unit_cnt = 0, gs = 0;
      bool ok = true;
      // S^T and dP^T of global step g into buffer g & 1.
      auto issue_s = [&](uint32_t g) -> bool {
        const int st = g % C::QSTAGE;
        if (!mbar_wait_bounded(bar(KB_QD_FULL + st), (g / C::QSTAGE) & 1, tmo, f.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t sq = sQD + st * C::STAGE_BYTES;
        const uint32_t b = g & 1;
        mma_s<D>(tmem + C::TM_S + 64 * b, sK, sq);                // S^T = K Q^T
        mma_s<D>(tmem + C::TM_DP + 64 * b, sV, sq + C::TILE64);   // dP^T = V dO^T
        tc_commit(bar(KB_S_FULL + b));
        return true;
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
        const KVUnit w = kv_unit(f, u);
        if (!mbar_wait_bounded(bar(KB_KV_FULL), unit_cnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (w.n_steps > 0 && !issue_s(gs)) { ok = false; break; }
        // The previous unit's accumulators must have been read out.
        if (unit_cnt > 0 &&
            !mbar_wait_bounded(bar(KB_ACC_EMPTY), (unit_cnt - 1) & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        for (int n = 0; n < w.n_steps; ++n) {
          const uint32_t g = gs + n;
          if (n + 1 < w.n_steps && !issue_s(g + 1)) { ok = false; break; }
          const uint32_t b = g & 1;
          if (!mbar_wait_bounded(bar(KB_P_FULL + b), (g >> 1) & 1, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sq = sQD + (g % C::QSTAGE) * C::STAGE_BYTES;
          mma_acc<D>(tdV, tmem + C::TM_S + 64 * b, sq + C::TILE64, n > 0);  // dV += P^T dO
          mma_acc<D>(tdK, tmem + C::TM_DP + 64 * b, sq, n > 0);            // dK += dS^T Q
          tc_commit(bar(KB_QD_EMPTY + g % C::QSTAGE));
        }
        if (!ok) break;
        gs += w.n_steps;
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
    const int wg = (warp - 4) >> 2;  // warpgroup: takes the steps g with g & 1 == wg
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tAcc = tmem + lane_off + (wg == 0 ? C::TM_DV : C::TM_DK);
    uint16_t* const out = static_cast<uint16_t*>(wg == 0 ? a.dv : a.dk);
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, gs = 0;
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
      for (int n = 0; n < w.n_steps; ++n) {
        const uint32_t g = gs + n;
        const uint32_t b = g & 1;
        if (static_cast<int>(b) != wg) continue;
        const int st = g % C::QSTAGE;
        const int q0 = w.qa + NSTEP * (n / G);
        bool e = mbar_wait_bounded(bar(KB_S_FULL + b), (g >> 1) & 1, tmo, f.err, abort_flag);
        e = e && mbar_wait_bounded(bar(KB_QD_FULL + st), (g / C::QSTAGE) & 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_QD + st * C::STAGE_BYTES + 2 * C::TILE64);
        const float* dd = lse2 + NSTEP;
        const int clo = kvalid ? max(lo, q0) - q0 : 0;
        const int chi = kvalid ? min(hi, q0 + NSTEP) - q0 : 0;
        const uint32_t tS = tmem + lane_off + C::TM_S + 64 * b;
        const uint32_t tdP = tmem + lane_off + C::TM_DP + 64 * b;
        grad_step<true>(tS, tdP, tdP, clo, chi, sl2, scale, [&](int c) { return lse2[c]; },
                        [&](int c) { return dd[c]; });
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_P_FULL + b));
      }
      if (!ok) break;
      gs += w.n_steps;
      const bool e = mbar_wait_bounded(bar(KB_ACC_FULL), unit_cnt & 1, tmo, f.err, abort_flag);
      if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
      tc_fence_after();
      // Warpgroup 0 writes dV, warpgroup 1 dK.
      const bool has_acc = w.n_steps > 0;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t rv[32];
        if (has_acc) tmem_ld32_sync(tAcc + 32 * ch, rv);
        if (kvalid) {
          uint16_t* dst = out + (static_cast<size_t>(j) * f.Hkv + w.hk) * D + 32 * ch;
          if (has_acc) store_row32_bf16(dst, rv);
          else store_zero_row_bf16(dst, 32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_ACC_EMPTY));
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
  static constexpr int KSTAGE = 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = B::TILE128;
  static constexpr int OFF_KV = 2 * B::TILE128;  // stage s: K at +0, V at +TILE64
  static constexpr int OFF_BAR = OFF_KV + KSTAGE * 2 * B::TILE64;
  static constexpr int N_BARS = 17;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DQ = 256;
};

enum { QB_Q_FULL = 0, QB_Q_EMPTY = 1, QB_KV_FULL = 2, QB_KV_EMPTY = 6, QB_S_FULL = 10, QB_P_FULL = 12,
       QB_ACC_FULL = 14, QB_DRAIN = 15, QB_ACC_EMPTY = 16 };

// Key steps of 64 over a unit's items for one Q tile: the forward's cursor
// (item key ranges clipped to the keys the tile's rows may attend) walked in
// 64-key blocks. full = every (row, key) of the block is valid.
__device__ __forceinline__ bool next_block64(const AttnArgs& a, Cursor& c, const QTile& qt, int& ka,
                                             int& kb, bool& full) {
  while (true) {
    if (c.k0 >= c.kv_e) {
      if (c.item >= c.item_end) return false;
      int b, e;
      item_range(a, c.item, b, e);
      ++c.item;
      c.k0 = max(b, c.lo);
      c.kv_e = min(e, c.hi);
      continue;
    }
    ka = c.k0;
    kb = min(c.k0 + NSTEP, c.kv_e);
    c.k0 += NSTEP;
    if (a.causal && ka > qt.qb - 1) continue;
    if (qt.de <= ka || kb <= qt.ds) continue;
    full = qt.qb - qt.qa == 128 && kb - ka == NSTEP && qt.one_doc && ka >= qt.ds && kb <= qt.de &&
           (!a.causal || kb - 1 <= qt.qa);
    return true;
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
bwd_dq_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tmq,
              const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
              const __grid_constant__ CUtensorMap tmdo) {
  using C = QCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO, sKV = sbase + C::OFF_KV;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(QB_S_FULL + b), 1);
      mbar_init(bar(QB_P_FULL + b), 4);
    }
    mbar_init(bar(QB_ACC_FULL), 1);
    mbar_init(bar(QB_DRAIN), 1);
    mbar_init(bar(QB_ACC_EMPTY), 8);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kv_cnt = 0, unit_cnt = 0;
      int armed_q = 0, armed_kv[C::KSTAGE] = {0, 0, 0, 0};
      uint32_t par_q = 0, par_kv[C::KSTAGE] = {0, 0, 0, 0};
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
        const UnitInfo ui = unit_info(f, u);
        const QTile qt = make_qtile(f, ui, 0);
        const QTile qts[2] = {qt, QTile{0, 0, 0, 0, 0}};
        const int hk = ui.h / G;
        if (!mbar_wait_bounded(bar(QB_Q_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(QB_Q_FULL), 2 * C::TILE128);
        armed_q = 1;
        par_q = unit_cnt & 1;
        load_rows128<D>(sQ, &tmq, bar(QB_Q_FULL), ui.h, ui.q0, f.T);
        load_rows128<D>(sDO, &tmdo, bar(QB_Q_FULL), ui.h, ui.q0, f.T);
        Cursor cur = make_cursor(ui, qts, f.causal);
        int ka, kb;
        bool full;
        while (next_block64(f, cur, qt, ka, kb, full)) {
          const int st = kv_cnt % C::KSTAGE;
          const uint32_t ph = (kv_cnt / C::KSTAGE) & 1;
          if (!mbar_wait_bounded(bar(QB_KV_EMPTY + st), ph ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(QB_KV_FULL + st), 2 * C::TILE64);
          armed_kv[st] = 1;
          par_kv[st] = ph;
          const uint32_t skv = sKV + st * 2 * C::TILE64;
          load_rows64<D>(skv, &tmk, bar(QB_KV_FULL + st), hk, ka);
          load_rows64<D>(skv + C::TILE64, &tmv, bar(QB_KV_FULL + st), hk, ka);
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
      const uint32_t tdQ = tmem + C::TM_DQ;
      uint32_t kv_cnt = 0, unit_cnt = 0;
      bool ok = true;
      // S and dP of key block g into buffer g & 1.
      auto issue_s = [&](uint32_t g) -> bool {
        const int st = g % C::KSTAGE;
        if (!mbar_wait_bounded(bar(QB_KV_FULL + st), (g / C::KSTAGE) & 1, tmo, f.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t skv = sKV + st * 2 * C::TILE64;
        const uint32_t b = g & 1;
        mma_s<D>(tmem + C::TM_S + 64 * b, sQ, skv);                // S = Q K^T
        mma_s<D>(tmem + C::TM_DP + 64 * b, sDO, skv + C::TILE64);  // dP = dO V^T
        tc_commit(bar(QB_S_FULL + b));
        return true;
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
        const UnitInfo ui = unit_info(f, u);
        const QTile qt = make_qtile(f, ui, 0);
        const QTile qts[2] = {qt, QTile{0, 0, 0, 0, 0}};
        if (!mbar_wait_bounded(bar(QB_Q_FULL), unit_cnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // Count the unit's key blocks (the walk is cheap and identical in every role).
        int nblk = 0;
        {
          Cursor cur = make_cursor(ui, qts, f.causal);
          int ka, kb;
          bool full;
          while (next_block64(f, cur, qt, ka, kb, full)) ++nblk;
        }
        if (nblk > 0 && !issue_s(kv_cnt)) { ok = false; break; }
        if (unit_cnt > 0 &&
            !mbar_wait_bounded(bar(QB_ACC_EMPTY), (unit_cnt - 1) & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        for (int n = 0; n < nblk; ++n) {
          const uint32_t g = kv_cnt + n;
          if (n + 1 < nblk && !issue_s(g + 1)) { ok = false; break; }
          const uint32_t b = g & 1;
          if (!mbar_wait_bounded(bar(QB_P_FULL + b), (g >> 1) & 1, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_acc<D>(tdQ, tmem + C::TM_S + 64 * b, sKV + (g % C::KSTAGE) * 2 * C::TILE64, n > 0);  // dQ += dS K
          tc_commit(bar(QB_KV_EMPTY + g % C::KSTAGE));
        }
        if (!ok) break;
        kv_cnt += nblk;
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
    const int wg = (warp - 4) >> 2;  // warpgroup: takes the blocks g with g & 1 == wg
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tdQ = tmem + lane_off + C::TM_DQ;
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_cnt) {
      const UnitInfo ui = unit_info(f, u);
      const QTile qt = make_qtile(f, ui, 0);
      const QTile qts[2] = {qt, QTile{0, 0, 0, 0, 0}};
      const int t = ui.q0 + r;
      const bool valid = t >= qt.qa && t < qt.qb;
      int rds = 0, rde = 0;
      float lse2 = 0.f, di = 0.f;
      if (valid) {
        const int dd = doc_of(f.cu, f.ndocs, t);
        rds = __ldg(f.cu + dd);
        rde = __ldg(f.cu + dd + 1);
        lse2 = __ldg(a.lse + static_cast<size_t>(ui.h) * f.T + t) * LOG2E;
        di = __ldg(a.dvec + static_cast<size_t>(ui.h) * f.T + t);
      }
      const int rend = f.causal ? min(rde, t + 1) : rde;
      int nblk = 0;
      Cursor cur = make_cursor(ui, qts, f.causal);
      int ka, kb;
      bool full;
      while (next_block64(f, cur, qt, ka, kb, full)) {
        const uint32_t b = g & 1;
        if (static_cast<int>(b) != wg) {
          ++g;
          ++nblk;
          continue;
        }
        const bool e = mbar_wait_bounded(bar(QB_S_FULL + b), (g >> 1) & 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        int lo = 0, hi = NSTEP;
        if (!full) {
          lo = valid ? max(ka, rds) - ka : 0;
          hi = valid ? min(kb, rend) - ka : 0;
        }
        const uint32_t tS = tmem + lane_off + C::TM_S + 64 * b;
        const uint32_t tdP = tmem + lane_off + C::TM_DP + 64 * b;
        grad_step<false>(tS, tdP, tS, lo, hi, sl2, scale, [&](int) { return lse2; },
                         [&](int) { return di; });
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_P_FULL + b));
        ++g;
        ++nblk;
      }
      if (!ok) break;
      const bool e = mbar_wait_bounded(bar(QB_ACC_FULL), unit_cnt & 1, tmo, f.err, abort_flag);
      if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
      tc_fence_after();
      // Each warpgroup writes half of the dQ columns.
#pragma unroll 1
      for (int ch = wg * (D / 64); ch < (wg + 1) * (D / 64); ++ch) {
        uint32_t rq[32];
        if (nblk > 0) tmem_ld32_sync(tdQ + 32 * ch, rq);
        if (valid) {
          uint16_t* dst = static_cast<uint16_t*>(a.dq) + (static_cast<size_t>(t) * f.Hq + ui.h) * D + 32 * ch;
          if (nblk > 0) store_row32_bf16(dst, rq);
          else store_zero_row_bf16(dst, 32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QB_ACC_EMPTY));
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
  kern<<<grid, 384, Cfg::SMEM_ALLOC, st>>>(a, q, k, v, dout);
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
