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
//   bwd_rowdot   -scale D_i and -LSE_i log2(e) per (row, head) into the workspace.
//   bwd_dkdv     one unit per (key/value head, 128-key tile), head-major so
//                that the CTAs running at one time share the Q and dO of one
//                head group in L2. K and V stay in shared memory while every
//                128-row Q tile that can attend the keys streams through (all
//                query heads of the group). Keys sit on the tensor-memory
//                lanes: S^T = K Q^T and dP^T = V dO^T, then dV += P^T dO and
//                dK += dS^T Q with P^T and dS^T read from tensor memory.
//   bwd_dq       one unit per (128-row Q tile, query head), walking the same
//                schedule items as the forward in 128-key tiles: S = Q K^T,
//                dP = dO V^T, dQ += dS K with dS read from tensor memory.
// Every MMA is 128 x 128 x 16 (a 128 x 64 MMA costs as long as a 128 x 128
// one, so narrower steps would halve the tensor-core rate). The elementwise
// work of a step is split by columns between two compute warpgroups (64
// columns each, P kept in registers between the S and the dP phase), and the
// MMA lane interleaves (dV or nothing)(g), S(g+1), (dK or dQ)(g), dP(g+1):
// S(g+1) runs while the warpgroups turn dP(g) into dS(g), and dK/dQ(g) and
// dP(g+1) run while they turn S(g+1) into P. Each kernel: warp 0 TMA
// producer, warp 1 TMEM owner and MMA lane, warps 4-11 two compute
// warpgroups (one TMEM lane, i.e. one key or query row, per thread). Tensor maps use {64 dims, 1 head, 64 rows}
// boxes with 128-byte swizzle; a 128-row tile is two boxes, row r at r x 128
// bytes of each 64-dim sub-tile, the layout one 128-row box would give.

#include <cuda.h>

#include <cstring>

#include "sp_device.cuh"
#include "sp_tiles.cuh"

namespace sp {
namespace {

constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int KSUB = D / 64;        // 64-dim sub-tiles
  static constexpr int SUB = 128 * 128;      // bytes of a 128-row sub-tile
  static constexpr int BOX = 64 * 128;       // bytes of a 64-row box
  static constexpr int TILE = KSUB * SUB;    // bytes of a 128-row tile
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);  // both K-major
  static constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, D, 0, 1);  // B MN-major
  static constexpr int TMEM_COLS = 512;
};

// K-major operand descriptor (rows = M or N, 64 dims per 128-byte row).
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return smem_desc_sw128(addr, 16, 1024); }
// MN-major B operand over a 128-row tile: the next 64 columns of N start one
// sub-tile further on.
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr) { return smem_desc_sw128(addr, 128 * 128, 1024); }

// D/16 MMAs contracting over d: C[128 x 128] = A B^T, A and B 128-row K-major tiles.
template <int D>
__device__ __forceinline__ void mma_s(uint32_t d_t, uint32_t a_addr, uint32_t b_addr) {
  using C = BCfg<D>;
  const uint64_t a0 = desc_k(a_addr), b0 = desc_k(b_addr);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t o = static_cast<uint64_t>(((kk >> 2) * C::SUB + (kk & 3) * 32) >> 4);
    tc_mma_ss(d_t, a0 + o, b0 + o, C::IDESC_S, kk > 0 ? 1u : 0u);
  }
}

// 8 MMAs contracting over 128 rows: C[128 x D] (+)= A(tmem) B(128 rows x D,
// MN-major). A holds bf16 pairs in two 32-column halves of a 128-column
// region: rows 0-63 of the contraction in columns 0-31, rows 64-127 in
// columns 64-95 (each written by one compute warpgroup over the columns it
// read).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t d_t, uint32_t a_t, uint32_t b_addr, int acc) {
  using C = BCfg<D>;
  const uint64_t b0 = desc_mn(b_addr);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    tc_mma_ts(d_t, a_t + 8 * kk + (kk >= 4 ? 32 : 0), b0 + static_cast<uint64_t>(kk * (2048 >> 4)),
              C::IDESC_ACC, (acc || kk > 0) ? 1u : 0u);
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
    tma_load_3d(dst + s * C::SUB, m, bar, 64 * s, h, row0);
    tma_load_3d(dst + s * C::SUB + C::BOX, m, bar, 64 * s, h, row1);
  }
}

// 4-byte asynchronous copy global -> shared, counted on an mbarrier by
// cp_async_arrive (no increment of the barrier's expected count).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Loads 64 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t t, uint32_t (&x)[64]) {
  uint32_t a[32];
  tmem_ld32_sync(t, a);
#pragma unroll
  for (int c = 0; c < 32; ++c) x[c] = a[c];
  tmem_ld32_sync(t + 32, a);
#pragma unroll
  for (int c = 0; c < 32; ++c) x[32 + c] = a[c];
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Per-column values of a step (one per query column, staged in shared memory)
// or one per-row value broadcast to every column; pair4(c) gives the pairs
// for columns (c, c+1) and (c+2, c+3).
struct ColVals {
  const float* v;
  __device__ __forceinline__ void pair4(int c, uint64_t& p01, uint64_t& p23) const {
    const float4 q = *reinterpret_cast<const float4*>(v + c);
    p01 = f2_pack(q.x, q.y);
    p23 = f2_pack(q.z, q.w);
  }
};
struct RowVal {
  uint64_t v2;
  __device__ __forceinline__ void pair4(int, uint64_t& p01, uint64_t& p23) const { p01 = p23 = v2; }
};

// One compute warpgroup's half of a step (64 of the 128 columns, starting
// at column c0 of the operand): given S of those columns in p[], replaces it
// by P = 2^(S sl2 + nlse2) with nlse2 = -LSE log2 e on columns [lo, hi) (0
// elsewhere), in fp32.
template <bool kMask, typename Src>
__device__ __forceinline__ void p_half_impl(int c0, int lo, int hi, float sl2, Src nlse2, uint32_t (&p)[64]) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
  for (int c = 0; c < 64; c += 4) {
    const int cc = c0 + c;
    uint64_t n01, n23;
    nlse2.pair4(cc, n01, n23);
    const uint64_t a01 = f2_fma(f2_pack(__uint_as_float(p[c]), __uint_as_float(p[c + 1])), sl2x2, n01);
    const uint64_t a23 = f2_fma(f2_pack(__uint_as_float(p[c + 2]), __uint_as_float(p[c + 3])), sl2x2, n23);
    float e0, e1, e2, e3;
    f2_unpack(a01, e0, e1);
    f2_unpack(a23, e2, e3);
    float p0 = ex2_approx(e0), p1 = ex2_approx(e1), p2 = ex2_approx(e2), p3 = ex2_approx(e3);
    if (kMask) {
      p0 = (cc >= lo && cc < hi) ? p0 : 0.f;
      p1 = (cc + 1 >= lo && cc + 1 < hi) ? p1 : 0.f;
      p2 = (cc + 2 >= lo && cc + 2 < hi) ? p2 : 0.f;
      p3 = (cc + 3 >= lo && cc + 3 < hi) ? p3 : 0.f;
    }
    p[c] = __float_as_uint(p0);
    p[c + 1] = __float_as_uint(p1);
    p[c + 2] = __float_as_uint(p2);
    p[c + 3] = __float_as_uint(p3);
  }
}

// The mask is skipped when no lane of the warp needs it for these columns
// (the tensor-memory accesses must stay warp-uniform).
template <typename Src>
__device__ __forceinline__ void p_half(int c0, int lo, int hi, float sl2, Src nlse2, uint32_t (&p)[64]) {
  if (__all_sync(0xffffffffu, lo <= c0 && hi >= c0 + 64)) p_half_impl<false>(c0, lo, hi, sl2, nlse2, p);
  else p_half_impl<true>(c0, lo, hi, sl2, nlse2, p);
}

// 64 fp32 values as 32 bf16 pairs into 32 tensor-memory columns.
__device__ __forceinline__ void store_pairs32(uint32_t dst, const uint32_t (&v)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]));
  tmem_st32(dst, pk);
}

// dS = P (dP scale + ndsc) with ndsc = -D scale, i.e. P (dP - D) scale, for
// the same 64 columns (dP at t_dp, column c0 of the operand), written as 32
// bf16-pair columns at t_dp: chunk h of 32 dP columns writes packed columns
// 16h .. 16h+15, which chunk 0 has already read.
template <typename Src>
__device__ __forceinline__ void ds_half(uint32_t t_dp, int c0, const uint32_t (&p)[64], float scale, Src ndsc) {
  const uint64_t sc2 = f2_pack(scale, scale);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t dp[32];
    tmem_ld32_sync(t_dp + 32 * hh, dp);
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const int q = 32 * hh + c;
      uint64_t n01, n23;
      ndsc.pair4(c0 + q, n01, n23);
      const uint64_t t01 = f2_fma(f2_pack(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), sc2, n01);
      const uint64_t t23 = f2_fma(f2_pack(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3])), sc2, n23);
      const uint64_t d01 = f2_mul(f2_pack(__uint_as_float(p[q]), __uint_as_float(p[q + 1])), t01);
      const uint64_t d23 = f2_mul(f2_pack(__uint_as_float(p[q + 2]), __uint_as_float(p[q + 3])), t23);
      float s0, s1, s2, s3;
      f2_unpack(d01, s0, s1);
      f2_unpack(d23, s2, s3);
      pk[c >> 1] = pack_bf16x2(s0, s1);
      pk[(c >> 1) + 1] = pack_bf16x2(s2, s3);
    }
    tmem_st16(t_dp + 16 * hh, pk);
  }
}

// ------------------------------------------------------------------ D_i

// ndsc[h][t] = -scale * (dO[t][h][:] . O[t][h][:]) in fp32 from bf16, and
// nlse2[h][t] = -lse[h][t] * log2(e); one warp per (t, h). The signs and the
// scale are folded in so that the tensor-core kernels need one FMA per value.
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ dout,
                                                         const float* __restrict__ lse,
                                                         float* __restrict__ ndsc, float* __restrict__ nlse2,
                                                         int T, int Hq, int d, float scale) {
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
    if (lane == 0) {
      const size_t i = static_cast<size_t>(h) * T + t;
      ndsc[i] = -acc * scale;
      nlse2[i] = -lse[i] * LOG2E;
    }
  }
}

// ------------------------------------------------------------------ dK, dV

template <int D>
struct KVCfg : BCfg<D> {
  using B = BCfg<D>;
  static constexpr int QSTAGE = 2;
  static constexpr int STAGE_BYTES = 2 * B::TILE + 1024;  // Q, dO, LSE2[128], D[128]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = B::TILE;
  static constexpr int OFF_QD = 2 * B::TILE;
  static constexpr int OFF_BAR = OFF_QD + QSTAGE * STAGE_BYTES;
  static constexpr int N_BARS = 17;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;  // TMEM address, abort flag, unit ring[2]
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
};

enum { KB_KV_FULL = 0, KB_KV_EMPTY = 1, KB_QD_FULL = 2, KB_QD_EMPTY = 4, KB_S_FULL = 6, KB_DP_FULL = 7,
       KB_P_FULL = 8, KB_DS_FULL = 9, KB_ACC_FULL = 10, KB_ACC_EMPTY = 11, KB_DRAIN = 12, KB_U_FULL = 13,
       KB_U_EMPTY = 15 };
constexpr int KV_UNIT_CONSUMERS = 9;  // the MMA lane and the eight compute warps

struct KVUnit {
  int k0, k1, hk;  // keys [k0, k1) of key/value head hk
  int qa, qb;      // queries that may attend them
  int n_steps;     // 128-row Q tiles in [qa, qb) times the heads of the group
};

// Units are head-major: all key tiles of head 0, then head 1, ...; within a
// head the key tiles in order, which for causal masks is longest first. CTAs
// claim units from an atomic counter in that order.
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
  w.n_steps = ((w.qb - w.qa + 127) / 128) * (a.Hq / a.Hkv);
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
  volatile int* uring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnArgs& f = a.fwd;

  if (threadIdx.x == 0) {
    mbar_init(bar(KB_KV_FULL), 1);
    mbar_init(bar(KB_KV_EMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(KB_U_FULL + s), 1);
      mbar_init(bar(KB_U_EMPTY + s), KV_UNIT_CONSUMERS);
    }
    for (int s = 0; s < C::QSTAGE; ++s) {
      mbar_init(bar(KB_QD_FULL + s), 32);  // one asynchronous arrival per producer lane
      mbar_init(bar(KB_QD_EMPTY + s), 1);
    }
    mbar_init(bar(KB_S_FULL), 1);
    mbar_init(bar(KB_DP_FULL), 1);
    mbar_init(bar(KB_P_FULL), 8);   // both compute warpgroups, one arrival per warp
    mbar_init(bar(KB_DS_FULL), 8);
    mbar_init(bar(KB_ACC_FULL), 1);
    mbar_init(bar(KB_ACC_EMPTY), 8);
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
    uint32_t unit_cnt = 0, gs = 0;
    int armed_kv = 0, armed_qd[C::QSTAGE] = {0, 0};
    uint32_t par_kv = 0, par_qd[C::QSTAGE] = {0, 0};
    bool ok = true;
    int uslot = 0;
    uint32_t uph = 0;
    for (;; ++unit_cnt) {
      // Claim the next unit and hand its id to the other roles (-1: done).
      int u = 0;
      bool pub = true;
      if (lane == 0) {
        u = atomicAdd(a.unit_counter, 1);
        if (u >= n_units) u = -1;
        pub = mbar_wait_bounded(bar(KB_U_EMPTY + uslot), uph ^ 1, tmo, f.err, abort_flag);
        if (pub) {
          uring[uslot] = u;
          mbar_arrive(bar(KB_U_FULL + uslot));
        }
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!__shfl_sync(0xffffffffu, pub ? 1 : 0, 0)) { ok = false; break; }
      if (++uslot == 2) { uslot = 0; uph ^= 1; }
      if (u < 0) break;
      const KVUnit w = kv_unit(f, u);
      bool got = true;
      if (lane == 0) {
        got = mbar_wait_bounded(bar(KB_KV_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag);
        if (got) {
          mbar_arrive_expect_tx(bar(KB_KV_FULL), 2 * C::TILE);
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
        const int q0 = w.qa + 128 * (step / G);
        const bool e = mbar_wait_bounded(bar(KB_QD_EMPTY + st), ph ^ 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        const uint32_t full = bar(KB_QD_FULL + st);
        const uint32_t sq = sQD + st * C::STAGE_BYTES;
        if (lane == 0) {
          mbar_expect_tx(full, 2 * C::TILE);
          load_rows128<D>(sq, &tmq, full, h, q0, f.T);
          load_rows128<D>(sq + C::TILE, &tmdo, full, h, q0, f.T);
          armed_qd[st] = 1;
          par_qd[st] = ph;
        }
        // -LSE log2 e and -D scale of the tile's rows (rows past T read row
        // T-1: masked).
        const size_t hb = static_cast<size_t>(h) * f.T;
        for (int idx = lane; idx < 128; idx += 32) {
          const int row = min(q0 + idx, f.T - 1);
          cp_async4(sq + 2 * C::TILE + 4 * idx, a.nlse2 + hb + row);
          cp_async4(sq + 2 * C::TILE + 512 + 4 * idx, a.ndsc + hb + row);
        }
        cp_async_arrive(full);
      }
    }
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      if (armed_kv) mbar_wait_bounded(bar(KB_KV_FULL), par_kv, 50000000ull, f.err, &no_abort);
      for (int s = 0; s < C::QSTAGE; ++s)
        if (armed_qd[s]) mbar_wait_bounded(bar(KB_QD_FULL + s), par_qd[s], 50000000ull, f.err, &no_abort);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA lane
    if (lane == 0) {
      const uint32_t tS = tmem + C::TM_S, tdP = tmem + C::TM_DP;
      const uint32_t tdV = tmem + C::TM_DV, tdK = tmem + C::TM_DK;
      uint32_t unit_cnt = 0, gs = 0;
      bool ok = true;
      int uslot = 0;
      uint32_t uph = 0;
      for (;; ++unit_cnt) {
        if (!mbar_wait_bounded(bar(KB_U_FULL + uslot), uph, tmo, f.err, abort_flag)) { ok = false; break; }
        const int u = uring[uslot];
        mbar_arrive(bar(KB_U_EMPTY + uslot));
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (u < 0) break;
        const KVUnit w = kv_unit(f, u);
        if (!mbar_wait_bounded(bar(KB_KV_FULL), unit_cnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (w.n_steps > 0) {
          if (!mbar_wait_bounded(bar(KB_QD_FULL + gs % C::QSTAGE), (gs / C::QSTAGE) & 1, tmo, f.err,
                                 abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sq = sQD + (gs % C::QSTAGE) * C::STAGE_BYTES;
          mma_s<D>(tS, sK, sq);              // S^T = K Q^T
          tc_commit(bar(KB_S_FULL));
          mma_s<D>(tdP, sV, sq + C::TILE);   // dP^T = V dO^T
          tc_commit(bar(KB_DP_FULL));
        }
        // The previous unit's accumulators must have been read out.
        if (unit_cnt > 0 &&
            !mbar_wait_bounded(bar(KB_ACC_EMPTY), (unit_cnt - 1) & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        for (int n = 0; n < w.n_steps; ++n) {
          const uint32_t g = gs + n;
          const uint32_t ph = g & 1;
          const bool more = n + 1 < w.n_steps;
          const uint32_t sq = sQD + (g % C::QSTAGE) * C::STAGE_BYTES;
          const uint32_t sq1 = sQD + ((g + 1) % C::QSTAGE) * C::STAGE_BYTES;
          if (!mbar_wait_bounded(bar(KB_P_FULL), ph, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_acc<D>(tdV, tS, sq + C::TILE, n > 0);  // dV += P^T dO
          if (more) {
            // S(g+1) overwrites P^T(g): dV(g) is issued before it, and both
            // warpgroups have read S(g) (they keep P in registers).
            if (!mbar_wait_bounded(bar(KB_QD_FULL + (g + 1) % C::QSTAGE), ((g + 1) / C::QSTAGE) & 1, tmo,
                                   f.err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            mma_s<D>(tS, sK, sq1);
            tc_commit(bar(KB_S_FULL));
          }
          if (!mbar_wait_bounded(bar(KB_DS_FULL), ph, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_acc<D>(tdK, tdP, sq, n > 0);  // dK += dS^T Q
          tc_commit(bar(KB_QD_EMPTY + g % C::QSTAGE));
          if (more) {
            mma_s<D>(tdP, sV, sq1 + C::TILE);
            tc_commit(bar(KB_DP_FULL));
          }
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
    const int wg = (warp - 4) >> 2;  // warpgroup: columns [64 wg, 64 wg + 64) of every step
    const int c0 = 64 * wg;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S, tdP = tmem + lane_off + C::TM_DP;
    const uint32_t tAcc = tmem + lane_off + (wg == 0 ? C::TM_DV : C::TM_DK);
    uint16_t* const out = static_cast<uint16_t*>(wg == 0 ? a.dv : a.dk);
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, gs = 0;
    bool ok = true;
    int uslot = 0;
    uint32_t uph = 0;
    for (;; ++unit_cnt) {
      const bool eu = mbar_wait_bounded(bar(KB_U_FULL + uslot), uph, tmo, f.err, abort_flag);
      if (!__all_sync(0xffffffffu, eu)) { ok = false; break; }
      const int u = uring[uslot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_U_EMPTY + uslot));
      if (++uslot == 2) { uslot = 0; uph ^= 1; }
      if (u < 0) break;
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
        const uint32_t ph = g & 1;
        const int q0 = w.qa + 128 * (n / G);
        const uint8_t* stage = smem + C::OFF_QD + (g % C::QSTAGE) * C::STAGE_BYTES + 2 * C::TILE;
        const uint32_t qd_bar = bar(KB_QD_FULL + g % C::QSTAGE), qd_ph = (g / C::QSTAGE) & 1;
        // Both warpgroups: P for query columns [c0, c0 + 64), packed into
        // S columns c0 .. c0+31; then dS for the same columns into dP.
        bool e = mbar_wait_bounded(bar(KB_S_FULL), ph, tmo, f.err, abort_flag);
        e = e && mbar_wait_bounded(qd_bar, qd_ph, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        const int clo = kvalid ? max(lo, q0) - q0 : 0;
        const int chi = kvalid ? min(hi, q0 + 128) - q0 : 0;
        uint32_t p[64];
        tmem_ld64(tS + c0, p);
        p_half(c0, clo, chi, sl2, ColVals{reinterpret_cast<const float*>(stage)}, p);
        store_pairs32(tS + c0, p);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_P_FULL));
        e = mbar_wait_bounded(bar(KB_DP_FULL), ph, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        ds_half(tdP + c0, c0, p, scale, ColVals{reinterpret_cast<const float*>(stage + 512)});
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_DS_FULL));
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
  // K tile g is read by S(g) and dQ(g), the last MMA of step g; V tile g only
  // by dP(g), issued a step earlier. So K has one stage more than V: the copy
  // of step g+3's K starts when dQ(g) is done and has a whole step to land.
  static constexpr int KSTAGE = 3;
  static constexpr int VSTAGE = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = B::TILE;
  static constexpr int OFF_K = 2 * B::TILE;
  static constexpr int OFF_V = OFF_K + KSTAGE * B::TILE;
  static constexpr int OFF_BAR = OFF_V + VSTAGE * B::TILE;
  static constexpr int N_BARS = 24;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int OFF_UREC = OFF_MISC + 16;  // two unit records
  static constexpr int SMEM_ALLOC = OFF_UREC + 2 * 64 + 1024;
  static constexpr int TM_S = 0, TM_DP = 128, TM_DQ = 256;
};

// KV_FULL[s] completes when K stage s and the V tile loaded with it have landed.
enum { QB_Q_FULL = 0, QB_Q_EMPTY = 1, QB_KV_FULL = 2, QB_K_EMPTY = 5, QB_V_EMPTY = 8, QB_S_FULL = 10,
       QB_DP_FULL = 11, QB_S_READ = 12, QB_DS_FULL = 13, QB_ACC_FULL = 14, QB_ACC_EMPTY = 15,
       QB_DRAIN = 16, QB_U_FULL = 17, QB_U_EMPTY = 19 };

// dQ unit record (int32 words; slot stride 16 words): what every role needs to
// run a unit, built once by the scheduler warp: the unit (< 0: no more work),
// its query head and first row, its Q tile (bounds and documents), the cursor
// standing on its first key tile, and the number of key tiles.
enum { DR_V = 0, DR_H = 1, DR_Q0 = 2, DR_QT = 3, DR_CUR = 8, DR_NBLK = 14, DR_N = 15 };
constexpr int DQ_UNIT_CONSUMERS = 10;  // producer, MMA lane, eight compute warps

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
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO;
  auto sk = [&](uint32_t g) { return sbase + C::OFF_K + (g % C::KSTAGE) * C::TILE; };
  auto sv = [&](uint32_t g) { return sbase + C::OFF_V + (g % C::VSTAGE) * C::TILE; };
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* urec = reinterpret_cast<volatile int*>(smem + C::OFF_UREC);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(QB_Q_FULL), 1);
    mbar_init(bar(QB_Q_EMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(QB_U_FULL + s), 1);
      mbar_init(bar(QB_U_EMPTY + s), DQ_UNIT_CONSUMERS);
    }
    for (int s = 0; s < C::KSTAGE; ++s) {
      mbar_init(bar(QB_KV_FULL + s), 1);
      mbar_init(bar(QB_K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::VSTAGE; ++s) mbar_init(bar(QB_V_EMPTY + s), 1);
    mbar_init(bar(QB_S_FULL), 1);
    mbar_init(bar(QB_DP_FULL), 1);
    mbar_init(bar(QB_S_READ), 8);   // both compute warpgroups, one arrival per warp
    mbar_init(bar(QB_DS_FULL), 8);
    mbar_init(bar(QB_ACC_FULL), 1);
    mbar_init(bar(QB_ACC_EMPTY), 8);
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

  // Units reach every role as records in a two-slot ring (see DR_*). Reads
  // one (the caller arrives on its slot's EMPTY barrier afterwards): false on
  // a timeout. The unit's single Q tile is qt[0]; qt[1] stays empty.
  auto read_unit = [&](int slot, uint32_t ph, int& v, int& h, int& q0, QTile (&qt)[2], Cursor& cur,
                       int& nblk) -> bool {
    if (!mbar_wait_bounded(bar(QB_U_FULL + slot), ph, tmo, f.err, abort_flag)) return false;
    const volatile int* rs = urec + 16 * slot;
    v = rs[DR_V];
    if (v < 0) return true;
    h = rs[DR_H];
    q0 = rs[DR_Q0];
    qt[0].qa = rs[DR_QT + 0];
    qt[0].qb = rs[DR_QT + 1];
    qt[0].ds = rs[DR_QT + 2];
    qt[0].de = rs[DR_QT + 3];
    qt[0].one_doc = rs[DR_QT + 4];
    qt[1].qa = qt[1].qb = qt[1].ds = qt[1].de = qt[1].one_doc = 0;
    cur.item = rs[DR_CUR + 0];
    cur.item_end = rs[DR_CUR + 1];
    cur.kv_e = rs[DR_CUR + 2];
    cur.k0 = rs[DR_CUR + 3];
    cur.lo = rs[DR_CUR + 4];
    cur.hi = rs[DR_CUR + 5];
    nblk = rs[DR_NBLK];
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kv_cnt = 0, unit_cnt = 0;
      int armed_q = 0, armed_kv[C::KSTAGE] = {};
      uint32_t par_q = 0, par_kv[C::KSTAGE] = {};
      bool ok = true;
      for (;; ++unit_cnt) {
        int v = -1, h = 0, q0 = 0, nblk = 0;
        QTile qt[2];
        Cursor cur;
        if (!read_unit(unit_cnt & 1, (unit_cnt >> 1) & 1, v, h, q0, qt, cur, nblk)) { ok = false; break; }
        mbar_arrive(bar(QB_U_EMPTY + (unit_cnt & 1)));
        if (v < 0) break;
        const int hk = h / G;
        if (!mbar_wait_bounded(bar(QB_Q_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(QB_Q_FULL), 2 * C::TILE);
        armed_q = 1;
        par_q = unit_cnt & 1;
        load_rows128<D>(sQ, &tmq, bar(QB_Q_FULL), h, q0, f.T);
        load_rows128<D>(sDO, &tmdo, bar(QB_Q_FULL), h, q0, f.T);
        int ka, kb, cls[2];
        while (next_tile(f, cur, qt, ka, kb, cls)) {
          const int st = kv_cnt % C::KSTAGE, vs = kv_cnt % C::VSTAGE;
          const uint32_t ph = (kv_cnt / C::KSTAGE) & 1, vph = (kv_cnt / C::VSTAGE) & 1;
          if (!mbar_wait_bounded(bar(QB_K_EMPTY + st), ph ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
          if (!mbar_wait_bounded(bar(QB_V_EMPTY + vs), vph ^ 1, tmo, f.err, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(QB_KV_FULL + st), 2 * C::TILE);
          armed_kv[st] = 1;
          par_kv[st] = ph;
          load_rows128<D>(sk(kv_cnt), &tmk, bar(QB_KV_FULL + st), hk, ka, f.T);
          load_rows128<D>(sv(kv_cnt), &tmv, bar(QB_KV_FULL + st), hk, ka, f.T);
          ++kv_cnt;
        }
        if (!ok) break;
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
      const uint32_t tS = tmem + C::TM_S, tdP = tmem + C::TM_DP, tdQ = tmem + C::TM_DQ;
      uint32_t kv_cnt = 0, unit_cnt = 0;
      bool ok = true;
      for (;; ++unit_cnt) {
        int v = -1, h = 0, q0 = 0, nblk = 0;
        QTile qt[2];
        Cursor cur;
        if (!read_unit(unit_cnt & 1, (unit_cnt >> 1) & 1, v, h, q0, qt, cur, nblk)) { ok = false; break; }
        mbar_arrive(bar(QB_U_EMPTY + (unit_cnt & 1)));
        if (v < 0) break;
        if (!mbar_wait_bounded(bar(QB_Q_FULL), unit_cnt & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (nblk > 0) {
          const uint32_t g = kv_cnt;
          if (!mbar_wait_bounded(bar(QB_KV_FULL + g % C::KSTAGE), (g / C::KSTAGE) & 1, tmo, f.err,
                                 abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_s<D>(tS, sQ, sk(g));          // S = Q K^T
          tc_commit(bar(QB_S_FULL));
          mma_s<D>(tdP, sDO, sv(g));        // dP = dO V^T
          tc_commit(bar(QB_DP_FULL));
          tc_commit(bar(QB_V_EMPTY + g % C::VSTAGE));
        }
        if (unit_cnt > 0 &&
            !mbar_wait_bounded(bar(QB_ACC_EMPTY), (unit_cnt - 1) & 1, tmo, f.err, abort_flag)) { ok = false; break; }
        for (int n = 0; n < nblk; ++n) {
          const uint32_t g = kv_cnt + n;
          const uint32_t ph = g & 1;
          const bool more = n + 1 < nblk;
          if (more) {
            // Both warpgroups have read S(g): S may be overwritten.
            if (!mbar_wait_bounded(bar(QB_S_READ), ph, tmo, f.err, abort_flag)) { ok = false; break; }
            if (!mbar_wait_bounded(bar(QB_KV_FULL + (g + 1) % C::KSTAGE), ((g + 1) / C::KSTAGE) & 1, tmo,
                                   f.err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            mma_s<D>(tS, sQ, sk(g + 1));
            tc_commit(bar(QB_S_FULL));
          }
          if (!mbar_wait_bounded(bar(QB_DS_FULL), ph, tmo, f.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          mma_acc<D>(tdQ, tdP, sk(g), n > 0);  // dQ += dS K
          tc_commit(bar(QB_K_EMPTY + g % C::KSTAGE));
          if (more) {
            mma_s<D>(tdP, sDO, sv(g + 1));
            tc_commit(bar(QB_DP_FULL));
            tc_commit(bar(QB_V_EMPTY + (g + 1) % C::VSTAGE));
          }
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
  } else if (warp == 2) {
    // ------------------------------------------------------------ unit scheduler
    // Claims units (from the set-up kernel's queue, largest groups first, or
    // strided over the CTAs) and builds each one's record ahead of the other
    // roles: the table searches and the walk over the unit's items (to count
    // its key tiles and find the first) are off their path.
    if (lane == 0) {
      int k_static = 0;
      for (uint32_t cnt = 0;; ++cnt) {
        int v;
        if (f.work_counter) {
          v = atomicAdd(f.work_counter, 1);
        } else {
          v = static_cast<int>(blockIdx.x) + k_static * static_cast<int>(gridDim.x);
          ++k_static;
        }
        if (v >= n_units) v = -1;
        int w[DR_N];
        w[DR_V] = v;
        if (v >= 0) {
          const UnitInfo ui = unit_info(f, v);
          QTile qt[2];
          qt[0] = make_qtile(f, ui, 0);
          qt[1].qa = qt[1].qb = qt[1].ds = qt[1].de = qt[1].one_doc = 0;
          Cursor cur = make_cursor(f, ui, qt, f.causal);
          Cursor walk = cur;
          int ka, kb, cls[2], nblk = 0;
          while (next_tile(f, walk, qt, ka, kb, cls)) {
            if (nblk == 0) {
              cur = walk;
              cur.k0 = ka;  // standing on the first tile
            }
            ++nblk;
          }
          w[DR_H] = ui.h;
          w[DR_Q0] = ui.q0;
          w[DR_QT + 0] = qt[0].qa;
          w[DR_QT + 1] = qt[0].qb;
          w[DR_QT + 2] = qt[0].ds;
          w[DR_QT + 3] = qt[0].de;
          w[DR_QT + 4] = qt[0].one_doc;
          w[DR_CUR + 0] = cur.item;
          w[DR_CUR + 1] = cur.item_end;
          w[DR_CUR + 2] = cur.kv_e;
          w[DR_CUR + 3] = cur.k0;
          w[DR_CUR + 4] = cur.lo;
          w[DR_CUR + 5] = cur.hi;
          w[DR_NBLK] = nblk;
        }
        const int slot = cnt & 1;
        if (!mbar_wait_bounded(bar(QB_U_EMPTY + slot), ((cnt >> 1) & 1) ^ 1, tmo, f.err, abort_flag)) break;
        volatile int* rs = urec + 16 * slot;
        const int n = v >= 0 ? static_cast<int>(DR_N) : 1;
        for (int i = 0; i < n; ++i) rs[i] = w[i];
        mbar_arrive(bar(QB_U_FULL + slot));
        if (v < 0) break;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    const int wg = (warp - 4) >> 2;  // warpgroup: columns [64 wg, 64 wg + 64) of every block
    const int c0 = 64 * wg;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S, tdP = tmem + lane_off + C::TM_DP;
    const uint32_t tdQ = tmem + lane_off + C::TM_DQ;
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, g = 0;
    bool ok = true;
    for (;; ++unit_cnt) {
      int v = -1, h = 0, q0 = 0, nblk_u = 0;
      QTile qt[2];
      Cursor cur;
      const bool got = read_unit(unit_cnt & 1, (unit_cnt >> 1) & 1, v, h, q0, qt, cur, nblk_u);
      __syncwarp();
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      if (lane == 0) mbar_arrive(bar(QB_U_EMPTY + (unit_cnt & 1)));
      if (v < 0) break;
      const int t = q0 + r;
      const bool valid = t >= qt[0].qa && t < qt[0].qb;
      int rds = 0, rde = 0;
      float nlse2 = 0.f, ndsc = 0.f;
      if (valid) {
        if (qt[0].one_doc) {  // the tile's rows are all in one document
          rds = qt[0].ds;
          rde = qt[0].de;
        } else {
          const int dd = doc_of(f.cu, f.ndocs, t);
          rds = __ldg(f.cu + dd);
          rde = __ldg(f.cu + dd + 1);
        }
        nlse2 = __ldg(a.nlse2 + static_cast<size_t>(h) * f.T + t);
        ndsc = __ldg(a.ndsc + static_cast<size_t>(h) * f.T + t);
      }
      const int rend = f.causal ? min(rde, t + 1) : rde;
      int nblk = 0;
      int ka, kb, cls[2];
      while (next_tile(f, cur, qt, ka, kb, cls)) {
        const uint32_t ph = g & 1;
        // Both warpgroups: P for key columns [c0, c0 + 64) in registers, then
        // dS for the same columns into dP.
        bool e = mbar_wait_bounded(bar(QB_S_FULL), ph, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        uint32_t p[64];
        tmem_ld64(tS + c0, p);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_S_READ));
        int lo = 0, hi = 128;
        if (cls[0] != CLS_FULL) {
          lo = valid ? max(ka, rds) - ka : 0;
          hi = valid ? min(kb, rend) - ka : 0;
        }
        p_half(c0, lo, hi, sl2, RowVal{f2_pack(nlse2, nlse2)}, p);
        e = mbar_wait_bounded(bar(QB_DP_FULL), ph, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        ds_half(tdP + c0, c0, p, scale, RowVal{f2_pack(ndsc, ndsc)});
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_DS_FULL));
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
          uint16_t* dst = static_cast<uint16_t*>(a.dq) + (static_cast<size_t>(t) * f.Hq + h) * D + 32 * ch;
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

cudaError_t launch_bwd_rowdot(const void* o, const void* dout, const float* lse, float* ndsc, float* nlse2,
                              int T, int Hq, int d, float scale, int grid, cudaStream_t st) {
  bwd_rowdot_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                         lse, ndsc, nlse2, T, Hq, d, scale);
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
