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
//   bwd_rowdot     -scale D_i and -LSE_i log2(e) per (row, head) into the
//                  workspace; zeroes the fp32 dQ accumulator and the unit queue.
//   bwd_fused      one unit per (key/value head, 128-key tile), head-major so
//                  that the CTAs running at one time share the Q, dO and dQ
//                  accumulator rows of one head group in L2. K and V stay in
//                  shared memory while every 128-row Q tile that can attend the
//                  keys streams through (all query heads of the group). Keys
//                  sit on the tensor-memory lanes: S^T = K Q^T, dP^T = V dO^T,
//                  dV += P^T dO and dK += dS^T Q with P^T and dS^T read from
//                  tensor memory; dS also goes to shared memory, where it is
//                  the B operand of the step's dQ tile, dQ^T = K^T dS^T
//                  (d on the tensor-memory lanes, queries on the columns). The
//                  tile is added into an fp32 accumulator with reductions in
//                  which each warp covers 32 consecutive floats of one query's
//                  row (one 128-byte line); they are spread over the next
//                  step's phases because the L2 accepts reductions at a
//                  bounded rate (about 6 TB/s measured on this GPU).
//                  Each S and dP is computed once: 10 d FLOP of tensor work per
//                  valid (query, key) pair and query head.
//   bwd_dq_convert the accumulator rounded to bf16 into dQ.
// Every MMA is 128 x 128 x 16 or 128 x d x 16 (a 128 x 64 MMA costs as long
// as a 128 x 128 one, so narrower steps would halve the tensor-core rate). The
// elementwise work of a step is split by columns between two compute
// warpgroups (64 columns each, P kept in registers between the S and the dP
// phase). Per step g the MMA lane issues dK(g), dQ(g), dV(g+1), dP(g+1),
// S(g+2): dV(g+1) fills the time the compute warps take to read dQ(g) out of
// the tensor-memory columns dP(g+1) reuses, and S(g+2) runs while they turn
// dP(g+1) into dS. The fp32 reductions make dQ's summation order vary from run
// to run (dK and dV are summed in a fixed order). Roles: warp 0 TMA producer, warp 1 TMEM owner and MMA
// lane, warps 4-11 two compute warpgroups (one TMEM lane, i.e. one key or
// query row, per thread). Tensor maps use {64 dims, 1 head, 64 rows} boxes
// with 128-byte swizzle; a 128-row tile is two boxes, row r at r x 128 bytes
// of each 64-dim sub-tile, the layout one 128-row box would give.

#include <cuda.h>

#include <cstring>
#include <type_traits>

#include "sp_device.cuh"

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
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, D == 128 ? 128 : D, 1, 1);  // A, B MN-major
  static constexpr int TMEM_COLS = 512;
};

// K-major operand descriptor (rows = M or N, 64 dims per 128-byte row).
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return smem_desc_sw128(addr, 16, 1024); }
// MN-major operand over a 128-row tile: the next 64 columns of M or N start
// one sub-tile further on.
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

// 8 MMAs contracting over the 128 keys of a tile. dS sits in shared memory
// as [key][query] (two 64-query sub-tiles, query-major); K is the key tile
// ([key][d], d-major).
// d = 128: dQ_tile^T[d x 128 queries] = K^T dS^T (A = K, B = dS), so that the
//   tensor-memory lanes are the head dimension and a warp's 32 lanes hold 32
//   consecutive floats of one query's accumulator row.
// d = 64: dQ_tile[128 queries x d] = dS K (a 64-row MMA would change the
//   tensor-memory layout; this head dimension is not on the fast path).
template <int D>
__device__ __forceinline__ void mma_dq(uint32_t d_t, uint32_t ds_addr, uint32_t k_addr) {
  using C = BCfg<D>;
  const uint64_t ds0 = desc_mn(ds_addr), k0 = desc_mn(k_addr);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t o = static_cast<uint64_t>(kk * (2048 >> 4));
    if (D == 128) tc_mma_ss(d_t, k0 + o, ds0 + o, C::IDESC_DQ, kk > 0 ? 1u : 0u);
    else tc_mma_ss(d_t, ds0 + o, k0 + o, C::IDESC_DQ, kk > 0 ? 1u : 0u);
  }
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Adds four consecutive fp32 values into global memory (p 16-byte aligned).
__device__ __forceinline__ void red_add_v4(float* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "f"(__uint_as_float(a)), "f"(__uint_as_float(b)), "f"(__uint_as_float(c)),
                  "f"(__uint_as_float(d))
               : "memory");
}
__device__ __forceinline__ void red_add(float* p, uint32_t a) {
  asm volatile("red.global.add.f32 [%0], %1;" :: "l"(p), "f"(__uint_as_float(a)) : "memory");
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

// Loads 64 consecutive TMEM columns of this thread's lane (one load, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t t, uint32_t (&x)[64]) { tmem_ld64_sync(t, x); }

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Per-column values of a step (one per query column, staged in shared memory);
// pair4(c) gives the pairs for columns (c, c+1) and (c+2, c+3).
struct ColVals {
  const float* v;
  __device__ __forceinline__ void pair4(int c, uint64_t& p01, uint64_t& p23) const {
    const float4 q = *reinterpret_cast<const float4*>(v + c);
    p01 = f2_pack(q.x, q.y);
    p23 = f2_pack(q.z, q.w);
  }
};

// One compute warpgroup's half of a step (64 of the 128 columns, starting
// at column c0 of the operand): given S of those columns in p[], replaces it
// by P = 2^(S sl2 + nlse2) with nlse2 = -LSE log2 e on columns [lo, hi) (0
// elsewhere), in fp32.
template <bool kMask>
__device__ __forceinline__ void p_half_impl(int c0, int lo, int hi, float sl2, ColVals nlse2, uint32_t (&p)[64]) {
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
__device__ __forceinline__ void p_half(int c0, int lo, int hi, float sl2, ColVals nlse2, uint32_t (&p)[64]) {
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
// the same 64 columns (dP at t_dp, column c0 of the operand), rounded to bf16
// pairs and written twice: over the first 32 of those tensor-memory columns
// (the A operand of dK += dS^T Q), and as this thread's 128-byte row of its
// warpgroup's 64-query sub-tile of dS in shared memory (the A operand of the
// dQ MMA), with the 128-byte swizzle: 16-byte chunk c of row r at chunk
// c ^ (r mod 8). Done in two halves of 32 columns (half hh writes packed
// columns 16hh .. 16hh+15, which half 0 has already read); between them
// mid() runs (the caller's other work).
template <typename Mid>
__device__ __forceinline__ void ds_half(uint32_t t_dp, int c0, const uint32_t (&p)[64], float scale,
                                        ColVals ndsc, uint32_t ds_row, uint32_t r7, Mid&& mid) {
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
#pragma unroll
    for (uint32_t ch = 0; ch < 4; ++ch)
      st_shared_v4(ds_row + (((4 * hh + ch) ^ r7) << 4), pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2],
                   pk[4 * ch + 3]);
    if (hh == 0) mid();
  }
}

// ------------------------------------------------------------------ D_i

// ndsc[h][t] = -scale * (dO[t][h][:] . O[t][h][:]) in fp32 from bf16, and
// nlse2[h][t] = -lse[h][t] * log2(e); d / 8 lanes per (t, h). The signs and the
// scale are folded in so that the tensor-core kernel needs one FMA per value.
// Also zeroes the (t, h) row of the fp32 dQ accumulator [T][Hq][d] and the
// fused kernel's unit counter, which the next kernel on the stream reads, and
// (block 0) checks the packing descriptor the masks come from: cu[0] = 0,
// strictly increasing, cu[ndocs] = T. A bad one sets *status, which makes the
// next two kernels write nothing (their row ranges come from it), and records
// ERR_INTERNAL.
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const uint16_t* __restrict__ o,
                                                         const uint16_t* __restrict__ dout,
                                                         const float* __restrict__ lse,
                                                         float* __restrict__ ndsc, float* __restrict__ nlse2,
                                                         float* __restrict__ dqacc, int32_t* unit_counter,
                                                         int32_t* status, const int32_t* __restrict__ cu,
                                                         int ndocs, unsigned* err, int T, int Hq, int d,
                                                         float scale) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0) {
    int bad = 0;
    for (int i = threadIdx.x; i <= ndocs; i += blockDim.x) {
      const int c = __ldg(cu + i);
      if ((i == 0 && c != 0) || (i == ndocs && c != T) || (i < ndocs && c >= __ldg(cu + i + 1))) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
      *unit_counter = 0;
      *status = bad;
      if (bad) atomicOr(err, ERR_INTERNAL_BIT);
    }
  }
  const long long n = static_cast<long long>(T) * Hq;
  // d / 8 lanes per (t, h) row, each with one 16-byte load of O and of dO
  // (elements [8 s, 8 s + 8) for sub-lane s), so that a warp takes 256 / d rows
  // at a time with every lane loading.
  const int lpr = d >> 3, rpw = 32 / lpr;
  const int sub = lane / lpr, sl = lane - sub * lpr;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5) * rpw;
  for (long long base = (static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * rpw;
       base < n; base += wstride) {
    const long long w = base + sub;
    const bool live = w < n;
    float acc = 0.f;
    if (live) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + static_cast<size_t>(w) * d) + sl);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + static_cast<size_t>(w) * d) + sl);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), acc);
        acc = fmaf(__uint_as_float(av[i] & 0xffff0000u), __uint_as_float(bv[i] & 0xffff0000u), acc);
      }
      float4* zq = reinterpret_cast<float4*>(dqacc + static_cast<size_t>(w) * d);
      zq[2 * sl] = make_float4(0.f, 0.f, 0.f, 0.f);
      zq[2 * sl + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // Sum over the row's lanes (xor offsets below lpr stay inside its segment).
    for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && sl == 0) {
      const int t = static_cast<int>(w / Hq), h = static_cast<int>(w % Hq);
      const size_t i = static_cast<size_t>(h) * T + t;
      ndsc[i] = -acc * scale;
      nlse2[i] = -lse[i] * LOG2E;
    }
  }
}

// dq = bf16(acc), 8 elements per thread and pass (n8 = elements / 8).
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                             uint16_t* __restrict__ dq, long long n8,
                                                             const int32_t* status) {
  if (*status) return;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 y = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    uint4 w;
    w.x = pack_bf16x2(x.x, x.y);
    w.y = pack_bf16x2(x.z, x.w);
    w.z = pack_bf16x2(y.x, y.y);
    w.w = pack_bf16x2(y.z, y.w);
    reinterpret_cast<uint4*>(dq)[i] = w;
  }
}

// ------------------------------------------------------------------ dK, dV, dQ

template <int D>
struct FCfg : BCfg<D> {
  using B = BCfg<D>;
  static constexpr int QSTAGE = 2;
  static constexpr int STAGE_BYTES = 2 * B::TILE + 1024;  // Q, dO, -LSE log2 e [128], -scale D [128]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = B::TILE;
  static constexpr int OFF_DS = 2 * B::TILE;  // dS [128 keys][128 queries] bf16: two 64-query sub-tiles
  static constexpr int OFF_QD = OFF_DS + 2 * B::SUB;
  static constexpr int OFF_BAR = OFF_QD + QSTAGE * STAGE_BYTES;
  static constexpr int N_BARS = 19;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;  // TMEM address, abort flag, unit ring[2]
  // The dynamic shared memory base is 1024-byte aligned on this GPU (the
  // kernel checks it), so the layout needs no slack for realignment: at
  // d = 128 it takes 231,600 of the 232,448 bytes a block may have.
  static constexpr int SMEM_ALLOC = OFF_MISC + 16;
  // Tensor memory: S^T (P^T as bf16 over its columns 0-31 and 64-95), dP^T
  // (then dS^T the same way), dV, dK. The dQ tile of a step takes the dP^T
  // columns at d = 128 (free once dS^T has been read by dK; lanes = d, columns
  // = queries) and columns of its own at d = 64 (lanes = queries).
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr int TM_DQ = D == 128 ? TM_DP : 256 + 2 * D;
  static constexpr int DQ_COLS = 64 * D / 128;  // dQ tile columns per compute warpgroup
};
static_assert(FCfg<128>::SMEM_ALLOC <= 232448, "fused backward layout exceeds the shared memory of a block");

enum { FB_KV_FULL = 0, FB_KV_EMPTY = 1, FB_QD_FULL = 2, FB_QD_EMPTY = 4, FB_S_FULL = 6, FB_DP_FULL = 7,
       FB_P_FULL = 8, FB_DS_FULL = 9, FB_DQ_FULL = 10, FB_DQ_READ = 11, FB_ACC_FULL = 12,
       FB_ACC_EMPTY = 13, FB_DRAIN = 14, FB_U_FULL = 15, FB_U_EMPTY = 17 };
constexpr int KV_UNIT_CONSUMERS = 9;  // the MMA lane and the eight compute warps

struct KVUnit {
  int k0, k1, hk;  // keys [k0, k1) of key/value head hk
  int qa, qb;      // queries that may attend them
  int n_steps;     // 128-row Q tiles in [qa, qb) times the heads of the group
};

// Units are head-major: all key tiles of head 0, then head 1, ...; within a
// head the key tiles in order, which for causal masks is longest first. CTAs
// claim units from an atomic counter in that order. Step n of a unit is query
// head hk G + n mod G over the Q tile at qa + 128 (n / G).
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
bwd_fused_kernel(const BwdArgs a, const __grid_constant__ CUtensorMap tmq,
                 const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const __grid_constant__ CUtensorMap tmdo) {
  using C = FCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const AttnArgs& f = a.fwd;
  if (*a.status) return;  // cu_seqlens failed the row-dot kernel's check: nothing is written
  if (sbase & 1023u) {  // the layout has no slack to realign (see FCfg)
    if (threadIdx.x == 0) atomicOr(f.err, ERR_INTERNAL_BIT);
    return;
  }
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
  const uint32_t sQD = sbase + C::OFF_QD;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* uring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(FB_KV_FULL), 1);
    mbar_init(bar(FB_KV_EMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(FB_U_FULL + s), 1);
      mbar_init(bar(FB_U_EMPTY + s), KV_UNIT_CONSUMERS);
    }
    for (int s = 0; s < C::QSTAGE; ++s) {
      mbar_init(bar(FB_QD_FULL + s), 32);  // one asynchronous arrival per producer lane
      mbar_init(bar(FB_QD_EMPTY + s), 1);
    }
    mbar_init(bar(FB_S_FULL), 1);
    mbar_init(bar(FB_DP_FULL), 1);
    mbar_init(bar(FB_P_FULL), 8);   // both compute warpgroups, one arrival per warp
    mbar_init(bar(FB_DS_FULL), 8);
    mbar_init(bar(FB_DQ_FULL), 1);
    mbar_init(bar(FB_DQ_READ), 8);
    mbar_init(bar(FB_ACC_FULL), 1);
    mbar_init(bar(FB_ACC_EMPTY), 8);
    mbar_init(bar(FB_DRAIN), 1);
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
  // Registers: the block is launched with 384 x 168; the producer/MMA
  // warpgroup gives up 48 per thread to the two compute warpgroups
  // (4 x 32 x 120 + 8 x 32 x 192 = 384 x 168).
  if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 120;");

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
        pub = mbar_wait_bounded(bar(FB_U_EMPTY + uslot), uph ^ 1, tmo, f.err, abort_flag);
        if (pub) {
          uring[uslot] = u;
          mbar_arrive(bar(FB_U_FULL + uslot));
        }
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (!__shfl_sync(0xffffffffu, pub ? 1 : 0, 0)) { ok = false; break; }
      if (++uslot == 2) { uslot = 0; uph ^= 1; }
      if (u < 0) break;
      const KVUnit w = kv_unit(f, u);
      bool got = true;
      if (lane == 0) {
        got = mbar_wait_bounded(bar(FB_KV_EMPTY), (unit_cnt & 1) ^ 1, tmo, f.err, abort_flag);
        if (got) {
          mbar_arrive_expect_tx(bar(FB_KV_FULL), 2 * C::TILE);
          armed_kv = 1;
          par_kv = unit_cnt & 1;
          load_rows128<D>(sK, &tmk, bar(FB_KV_FULL), w.hk, w.k0, f.T);
          load_rows128<D>(sV, &tmv, bar(FB_KV_FULL), w.hk, w.k0, f.T);
        }
      }
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) { ok = false; break; }
      for (int step = 0; step < w.n_steps; ++step, ++gs) {
        const int st = gs % C::QSTAGE;
        const uint32_t ph = (gs / C::QSTAGE) & 1;
        const int h = w.hk * G + step % G;
        const int q0 = w.qa + 128 * (step / G);
        const bool e = mbar_wait_bounded(bar(FB_QD_EMPTY + st), ph ^ 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        const uint32_t full = bar(FB_QD_FULL + st);
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
      if (!ok) break;
    }
    if (!ok && lane == 0) {
      volatile int no_abort = 0;
      if (armed_kv) mbar_wait_bounded(bar(FB_KV_FULL), par_kv, 50000000ull, f.err, &no_abort);
      for (int s = 0; s < C::QSTAGE; ++s)
        if (armed_qd[s]) mbar_wait_bounded(bar(FB_QD_FULL + s), par_qd[s], 50000000ull, f.err, &no_abort);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA lane
    if (lane == 0) {
      const uint32_t tS = tmem + C::TM_S, tdP = tmem + C::TM_DP;
      const uint32_t tdV = tmem + C::TM_DV, tdK = tmem + C::TM_DK, tdQ = tmem + C::TM_DQ;
      auto sq = [&](uint32_t g) { return sQD + (g % C::QSTAGE) * C::STAGE_BYTES; };
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait_bounded(bar(b), parity, tmo, f.err, abort_flag);
      };
      auto qd_ready = [&](uint32_t g) { return wait(FB_QD_FULL + g % C::QSTAGE, (g / C::QSTAGE) & 1); };
      uint32_t unit_cnt = 0, gs = 0;
      bool ok = true;
      int uslot = 0;
      uint32_t uph = 0;
      for (;; ++unit_cnt) {
        if (!wait(FB_U_FULL + uslot, uph)) { ok = false; break; }
        const int u = uring[uslot];
        mbar_arrive(bar(FB_U_EMPTY + uslot));
        if (++uslot == 2) { uslot = 0; uph ^= 1; }
        if (u < 0) break;
        const KVUnit w = kv_unit(f, u);
        if (!wait(FB_KV_FULL, unit_cnt & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t g0 = gs;
        const int ns = w.n_steps;
        if (ns > 0) {
          if (!qd_ready(g0)) { ok = false; break; }
          tc_fence_after();
          mma_s<D>(tS, sK, sq(g0));  // S^T = K Q^T
          tc_commit(bar(FB_S_FULL));
          // dP^T lands where the previous step's dQ tile was (d = 128).
          if (g0 > 0 && !wait(FB_DQ_READ, (g0 - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          mma_s<D>(tdP, sV, sq(g0) + C::TILE);  // dP^T = V dO^T
          tc_commit(bar(FB_DP_FULL));
        }
        // The previous unit's accumulators must have been read out.
        if (unit_cnt > 0 && !wait(FB_ACC_EMPTY, (unit_cnt - 1) & 1)) { ok = false; break; }
        if (ns > 0) {
          if (!wait(FB_P_FULL, g0 & 1)) { ok = false; break; }
          tc_fence_after();
          mma_acc<D>(tdV, tS, sq(g0) + C::TILE, 0);  // dV = P^T dO
          if (ns > 1) {
            if (!qd_ready(g0 + 1)) { ok = false; break; }
            tc_fence_after();
            mma_s<D>(tS, sK, sq(g0 + 1));  // overwrites P^T(g0) after dV(g0) read it
            tc_commit(bar(FB_S_FULL));
          }
        }
        for (int n = 0; n < ns; ++n) {
          const uint32_t g = g0 + n;
          if (!wait(FB_DS_FULL, g & 1)) { ok = false; break; }
          tc_fence_after();
          mma_acc<D>(tdK, tdP, sq(g), n > 0);  // dK += dS^T Q
          tc_commit(bar(FB_QD_EMPTY + g % C::QSTAGE));
          mma_dq<D>(tdQ, sDS, sK);  // dQ tile = dS K
          tc_commit(bar(FB_DQ_FULL));
          if (n + 1 < ns) {
            if (!wait(FB_P_FULL, (g + 1) & 1)) { ok = false; break; }
            tc_fence_after();
            mma_acc<D>(tdV, tS, sq(g + 1) + C::TILE, 1);  // dV += P^T dO
            if (!wait(FB_DQ_READ, g & 1)) { ok = false; break; }
            tc_fence_after();
            mma_s<D>(tdP, sV, sq(g + 1) + C::TILE);
            tc_commit(bar(FB_DP_FULL));
            if (n + 2 < ns) {
              if (!qd_ready(g + 2)) { ok = false; break; }
              tc_fence_after();
              mma_s<D>(tS, sK, sq(g + 2));
              tc_commit(bar(FB_S_FULL));
            }
          }
        }
        if (!ok) break;
        gs += ns;
        tc_commit(bar(FB_KV_EMPTY));
        tc_commit(bar(FB_ACC_FULL));
      }
      volatile int no_abort = 0;
      tc_commit(bar(FB_DRAIN));
      mbar_wait_bounded(bar(FB_DRAIN), 0, 50000000ull, f.err, &no_abort);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;");
    using B = BCfg<D>;
    const int wg = (warp - 4) >> 2;  // warpgroup: columns [64 wg, 64 wg + 64) of every step
    const int c0 = 64 * wg;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S, tdP = tmem + lane_off + C::TM_DP;
    const uint32_t tdQ = tmem + lane_off + C::TM_DQ + C::DQ_COLS * wg;
    const uint32_t tAcc = tmem + lane_off + (wg == 0 ? C::TM_DV : C::TM_DK);
    uint16_t* const out = static_cast<uint16_t*>(wg == 0 ? a.dv : a.dk);
    // This thread's row (key r) of its warpgroup's 64-query sub-tile of dS.
    const uint32_t ds_row = sDS + wg * B::SUB + r * 128;
    const uint32_t r7 = static_cast<uint32_t>(r & 7);
    const float sl2 = f.scale_log2, scale = f.scale;
    uint32_t unit_cnt = 0, gs = 0;
    bool ok = true;
    int uslot = 0;
    uint32_t uph = 0;
    for (;; ++unit_cnt) {
      const bool eu = mbar_wait_bounded(bar(FB_U_FULL + uslot), uph, tmo, f.err, abort_flag);
      if (!__all_sync(0xffffffffu, eu)) { ok = false; break; }
      const int u = uring[uslot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(FB_U_EMPTY + uslot));
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
      // dQ tile of a step out of tensor memory. d = 128: this thread holds
      // dimension r of the warpgroup's 64 queries, and each warp-wide
      // reduction covers 32 consecutive floats of one query's accumulator row
      // (one 128-byte line). The 64 values are read at once (so that dP of the
      // next step can reuse the columns) and kept as pending reductions that
      // are issued in four groups of 16 spread over the next step's phases:
      // the L2 takes reductions at a bounded rate, and issued in one burst
      // they would hold up the warp.
      // d = 64: this thread holds 32 dimensions of query row r, reduced at once.
      uint32_t pend[64];
      float* pend_p = nullptr;
      int pend_nv = 0;  // columns whose query row exists (rows past the tile's last document receive nothing)
      const size_t rs = static_cast<size_t>(f.Hq) * D;
      auto flush = [&](auto lo_c, auto hi_c) {
        constexpr int LO = decltype(lo_c)::value, HI = decltype(hi_c)::value;
        if (pend_nv >= HI) {
#pragma unroll
          for (int c = LO; c < HI; ++c) red_add(pend_p + c * rs, pend[c]);
        } else {
#pragma unroll
          for (int c = LO; c < HI; ++c)
            if (c < pend_nv) red_add(pend_p + c * rs, pend[c]);
        }
      };
      using I0 = std::integral_constant<int, 0>;
      using I32 = std::integral_constant<int, 32>;
      using I48 = std::integral_constant<int, 48>;
      using I64 = std::integral_constant<int, 64>;
      auto dq_take = [&](uint32_t g, int n) -> bool {
        const bool e = mbar_wait_bounded(bar(FB_DQ_FULL), g & 1, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) return false;
        tc_fence_after();
        const int h = w.hk * G + n % G;
        if constexpr (D == 128) {
          const int tq = w.qa + 128 * (n / G) + 64 * wg;  // query of this warpgroup's first column
          tmem_ld64(tdQ, pend);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(FB_DQ_READ));
          pend_p = a.dqacc + (static_cast<size_t>(tq) * f.Hq + h) * D + r;
          pend_nv = w.qb - tq;
        } else {
          const int t = w.qa + 128 * (n / G) + r;
          float* dst = a.dqacc + (static_cast<size_t>(t) * f.Hq + h) * D + 32 * wg;
          uint32_t x[32];
          tmem_ld32_sync(tdQ, x);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(FB_DQ_READ));
          if (t < w.qb) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) red_add_v4(dst + i, x[i], x[i + 1], x[i + 2], x[i + 3]);
          }
        }
        return true;
      };
      for (int n = 0; n < w.n_steps; ++n) {
        const uint32_t g = gs + n;
        const uint32_t ph = g & 1;
        const int q0 = w.qa + 128 * (n / G);
        const uint8_t* stage = smem + C::OFF_QD + (g % C::QSTAGE) * C::STAGE_BYTES + 2 * C::TILE;
        const uint32_t qd_bar = bar(FB_QD_FULL + g % C::QSTAGE), qd_ph = (g / C::QSTAGE) & 1;
        if (D == 128 && n > 1) flush(I48{}, I64{});  // last group of step n-2's dQ tile
        // P for query columns [c0, c0 + 64), packed into S columns c0 .. c0+31.
        bool e = mbar_wait_bounded(bar(FB_S_FULL), ph, tmo, f.err, abort_flag);
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
        if (lane == 0) mbar_arrive(bar(FB_P_FULL));
        // The previous step's dQ tile, while dV(g) runs.
        if (n > 0) {
          if (!dq_take(g - 1, n - 1)) { ok = false; break; }
          if (D == 128) flush(I0{}, I32{});
        }
        // dS for the same columns: into dP (tensor memory) and dS (shared).
        e = mbar_wait_bounded(bar(FB_DP_FULL), ph, tmo, f.err, abort_flag);
        if (!__all_sync(0xffffffffu, e)) { ok = false; break; }
        tc_fence_after();
        ds_half(tdP + c0, c0, p, scale, ColVals{reinterpret_cast<const float*>(stage + 512)}, ds_row, r7,
                [&] {
                  if (D == 128 && n > 0) flush(I32{}, I48{});
                });
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(FB_DS_FULL));
      }
      if (!ok) break;
      if (D == 128 && w.n_steps > 1) flush(I48{}, I64{});
      if (w.n_steps > 0) {
        if (!dq_take(gs + w.n_steps - 1, w.n_steps - 1)) { ok = false; break; }
        if (D == 128) {
          flush(I0{}, I32{});
          flush(I32{}, I48{});
          flush(I48{}, I64{});
        }
      }
      gs += w.n_steps;
      const bool e = mbar_wait_bounded(bar(FB_ACC_FULL), unit_cnt & 1, tmo, f.err, abort_flag);
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
      if (lane == 0) mbar_arrive(bar(FB_ACC_EMPTY));
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
                              float* dqacc, int32_t* unit_counter, int32_t* status, const int32_t* cu,
                              int ndocs, unsigned* err, int T, int Hq, int d, float scale, int grid,
                              cudaStream_t st) {
  bwd_rowdot_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                         lse, ndsc, nlse2, dqacc, unit_counter, status, cu, ndocs, err, T, Hq,
                                         d, scale);
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
  cudaError_t e = a.fwd.d == 128
                      ? launch_cfg<FCfg<128>>(bwd_fused_kernel<128>, kv_grid, st, a, mq, mk, mv, mdo)
                      : launch_cfg<FCfg<64>>(bwd_fused_kernel<64>, kv_grid, st, a, mq, mk, mv, mdo);
  if (e != cudaSuccess) return e;
  const long long n8 = static_cast<long long>(a.fwd.T) * a.fwd.Hq * a.fwd.d / 8;
  long long cgrid = (n8 + 255) / 256;
  if (cgrid > static_cast<long long>(grid) * 8) cgrid = static_cast<long long>(grid) * 8;
  bwd_dq_convert_kernel<<<static_cast<int>(cgrid), 256, 0, st>>>(a.dqacc, static_cast<uint16_t*>(a.dq), n8,
                                                                a.status);
  return cudaGetLastError();
}

}  // namespace sp
