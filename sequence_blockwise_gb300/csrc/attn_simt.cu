// Blockwise packed attention in fp32 on the CUDA cores.
//
// The fp32 path exists for the fp32 tolerance (1e-5): tensor-core TF32 keeps a
// 10-bit mantissa, so fp32 inputs are multiplied and accumulated with FFMA.
// Same work units and schedule walk as the tensor-core kernel: a block owns 128
// query rows of one head, visits the group's items in schedule order, stages
// 32 keys at a time in shared memory, and merges each step into a running
// (max, sum, accumulator) with the log-sum-exp rule (HSAP abstract: partial
// attention; TASP abstract: every Q chunk reaches every KV chunk).

#include "sp_device.cuh"

namespace sp {
namespace {

constexpr int ROWS = 128;
constexpr int KCH = 32;

template <int D, int OUT_PARTIAL>
__global__ void __launch_bounds__(ROWS) attn_simt_kernel(const AttnArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;                 // [D][ROWS], transposed so each thread reads its own column
  float* Ks = Qs + D * ROWS;      // [KCH][D]
  float* Vs = Ks + KCH * D;       // [KCH][D]
  const int tid = threadIdx.x;
  const int n_units = n_units_of(a);
  const int G = a.Hq / a.Hkv;
  const float* __restrict__ q = static_cast<const float*>(a.q);
  const float* __restrict__ k = static_cast<const float*>(a.k);
  const float* __restrict__ v = static_cast<const float*>(a.v);
  const float NEG_INF = -__int_as_float(0x7f800000);

  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const UnitInfo ui = unit_info(a, u);
    const int hk = ui.h / G;
    const int t = ui.q0 + tid;
    const bool valid = t < ui.q_hi;
    const int q_last = min(ui.q0 + ROWS, ui.q_hi) - 1;
    int rds = 0, rde = 0;
    if (valid) {
      const int dd = doc_of(a.cu, a.ndocs, t);
      rds = __ldg(a.cu + dd);
      rde = __ldg(a.cu + dd + 1);
    }
    // Block-wide document span of the rows, for skipping key blocks.
    const int blk_ds = __ldg(a.cu + doc_of(a.cu, a.ndocs, ui.q0));
    const int blk_de = __ldg(a.cu + doc_of(a.cu, a.ndocs, q_last) + 1);

    __syncthreads();
    for (int idx = tid; idx < ROWS * D; idx += ROWS) {
      const int r = idx / D, c = idx % D;
      const int tt = ui.q0 + r;
      Qs[c * ROWS + r] = (tt < ui.q_hi) ? q[(static_cast<size_t>(tt) * a.Hq + ui.h) * D + c] : 0.f;
    }

    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    float m = NEG_INF, l = 0.f;

    for (int it = ui.item_lo; it < ui.item_hi; ++it) {
      int kvb, kve;
      item_range(a, it, kvb, kve);
      for (int k0 = kvb; k0 < kve; k0 += KCH) {
        const int kb = min(k0 + KCH, kve);
        if (a.causal && k0 > q_last) break;           // later keys are all in the future
        if (blk_de <= k0 || kb <= blk_ds) continue;   // no shared document
        __syncthreads();
        for (int idx = tid; idx < KCH * D; idx += ROWS) {
          const int j = idx / D, c = idx % D;
          const int kk = k0 + j;
          const size_t off = (static_cast<size_t>(kk) * a.Hkv + hk) * D + c;
          Ks[idx] = (kk < kb) ? k[off] : 0.f;
          Vs[idx] = (kk < kb) ? v[off] : 0.f;
        }
        __syncthreads();
        int lo = 0, hi = 0;
        if (valid) {
          lo = max(k0, rds) - k0;
          hi = min(min(kb, rde), a.causal ? t + 1 : kb) - k0;
        }
        float s[KCH];
#pragma unroll
        for (int j = 0; j < KCH; ++j) s[j] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
          const float qc = Qs[c * ROWS + tid];
#pragma unroll
          for (int j = 0; j < KCH; ++j) s[j] = fmaf(qc, Ks[j * D + c], s[j]);
        }
        float mt = NEG_INF;
#pragma unroll
        for (int j = 0; j < KCH; ++j) {
          s[j] = (j >= lo && j < hi) ? s[j] * a.scale : NEG_INF;
          mt = fmaxf(mt, s[j]);
        }
        const float m_new = fmaxf(m, mt);
        if (m_new == NEG_INF) continue;
        const float alpha = expf(m - m_new);
        l *= alpha;
#pragma unroll
        for (int c = 0; c < D; ++c) acc[c] *= alpha;
#pragma unroll
        for (int j = 0; j < KCH; ++j) {
          const float p = expf(s[j] - m_new);
          l += p;
#pragma unroll
          for (int c = 0; c < D; ++c) acc[c] = fmaf(p, Vs[j * D + c], acc[c]);
        }
        m = m_new;
      }
    }

    if (valid) {
      const bool live = l > 0.f;
      const float inv = live ? 1.f / l : 0.f;
      const float lse_v = live ? m + logf(l) : NEG_INF;
      float* dst;
      if (OUT_PARTIAL) {
        dst = static_cast<float*>(a.o) + (static_cast<size_t>(t - a.row_base) * a.Hq + ui.h) * D;
        a.lse[static_cast<size_t>(ui.h) * a.n_rows + (t - a.row_base)] = lse_v;
      } else {
        dst = static_cast<float*>(a.o) + (static_cast<size_t>(t) * a.Hq + ui.h) * D;
        a.lse[static_cast<size_t>(ui.h) * a.T + t] = lse_v;
      }
#pragma unroll
      for (int c = 0; c < D; c += 4)
        *reinterpret_cast<float4*>(dst + c) =
            make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
    }
  }
}

template <int D, int P>
cudaError_t launch_d(const AttnArgs& a, int grid, cudaStream_t st) {
  const size_t smem = sizeof(float) * (static_cast<size_t>(D) * ROWS + 2 * KCH * D);
  auto kern = attn_simt_kernel<D, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, ROWS, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, int grid, cudaStream_t st) {
  if (a.d == 128) return a.out_mode ? launch_d<128, 1>(a, grid, st) : launch_d<128, 0>(a, grid, st);
  return a.out_mode ? launch_d<64, 1>(a, grid, st) : launch_d<64, 0>(a, grid, st);
}

}  // namespace sp
