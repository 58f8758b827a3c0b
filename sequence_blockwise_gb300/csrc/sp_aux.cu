// Auxiliary kernels: the schedule set-up pass, the log-sum-exp merge of
// partials, and the bounded-wait self-test.

#include "sp_device.cuh"
#include "sp_workspace.h"

namespace sp {
namespace {

// Block-wide exclusive scan of one int64 per thread (1024 threads).
__device__ long long block_exclusive_scan(long long x, long long* tmp, long long* total) {
  const int tid = threadIdx.x;
  tmp[tid] = x;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const long long y = (tid >= off) ? tmp[tid - off] : 0;
    __syncthreads();
    tmp[tid] += y;
    __syncthreads();
  }
  const long long incl = tmp[tid];
  *total = tmp[1023];
  __syncthreads();
  return incl - x;
}

// Groups the items by (rank, Q range, head range) runs, estimates each
// group's cost as the 128-key tiles its items span (the walk of the group's
// longest unit), orders groups largest first, and assigns work-unit ranges.
// One block of 1024 threads. Also validates the items and head ranges.
__device__ __forceinline__ void item_heads_of(const int32_t* heads, int i, int Hq, int& h0, int& h1) {
  if (heads) {
    h0 = heads[2 * i];
    h1 = heads[2 * i + 1];
  } else {
    h0 = 0;
    h1 = Hq;
  }
}

// Does the item hold at least one (query, key) pair the document and causal
// masks allow? The documents that meet both its Q range and its key range are
// those from the later of the two ranges' first documents to the earlier of
// their last ones; the first with a valid pair ends the search. Every index
// stays in [0, nd] whatever cu holds.
__device__ bool item_has_pair(const int32_t* cu, int nd, int qb, int qe, int kb, int ke, int causal) {
  if (qb >= qe || kb >= ke) return false;
  const int d0 = max(doc_of(cu, nd, qb), doc_of(cu, nd, kb));
  const int d1 = min(doc_of(cu, nd, qe - 1), doc_of(cu, nd, ke - 1));
  for (int d = d0; d <= d1; ++d) {
    const int ds = __ldg(cu + d), de = __ldg(cu + d + 1);
    const int q0 = max(qb, ds), q1 = min(qe, de), k0 = max(kb, ds), k1 = min(ke, de);
    if (q0 < q1 && k0 < k1 && (!causal || k0 <= q1 - 1)) return true;
  }
  return false;
}

// Largest number of groups the set-up kernel orders and checks for overlap
// (the checks are quadratic in the group count); longer lists are rejected.
constexpr int MAX_GROUPS = SP_MAX_GROUPS;

__global__ void __launch_bounds__(1024)
prep_kernel(const sp_item* __restrict__ items, const int32_t* __restrict__ heads, int n, int T, int Hq,
            int Hkv, int rpu, int32_t* ws, unsigned* err, const int32_t* __restrict__ cu, int ndocs,
            int causal) {
  __shared__ long long scan_tmp[1024];
  __shared__ int bad;
  __shared__ int any_sorted;
  const WsLayout L = ws_layout(n);
  int32_t* header = ws;
  SegEntry* segs = reinterpret_cast<SegEntry*>(reinterpret_cast<char*>(ws) + L.off_segs);
  SegEntry* tmp = reinterpret_cast<SegEntry*>(reinterpret_cast<char*>(ws) + L.off_tmp);
  int32_t* starts = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + L.off_starts);
  long long* cost = reinterpret_cast<long long*>(reinterpret_cast<char*>(ws) + L.off_cost);
  const int tid = threadIdx.x;
  if (tid == 0) {
    bad = 0;
    any_sorted = 0;
  }
  __syncthreads();

  // The packing descriptor the masks come from: cu[0] = 0, strictly
  // increasing, cu[ndocs] = T (documents never overlap or run past the
  // sequence; HSAP abstract: no cross-contamination between packed documents).
  for (int i = tid; i <= ndocs; i += 1024) {
    const int c = __ldg(cu + i);
    if ((i == 0 && c != 0) || (i == ndocs && c != T) || (i < ndocs && c >= __ldg(cu + i + 1))) bad = 1;
  }
  const int chunk = (n + 1023) / 1024;
  const int i0 = min(n, tid * chunk), i1 = min(n, i0 + chunk);
  const int G = Hq / Hkv;
  // A new group starts where the rank, Q range or head range changes.
  auto starts_group = [&](int i) {
    if (i == 0) return true;
    const sp_item pv = items[i - 1], it = items[i];
    int a0, a1, b0, b1;
    item_heads_of(heads, i - 1, Hq, a0, a1);
    item_heads_of(heads, i, Hq, b0, b1);
    return pv.rank != it.rank || pv.q_begin != it.q_begin || pv.q_end != it.q_end || a0 != b0 || a1 != b1;
  };
  long long cnt = 0;
  for (int i = i0; i < i1; ++i) {
    const sp_item it = items[i];
    if (!(0 <= it.q_begin && it.q_begin < it.q_end && it.q_end <= T && 0 <= it.kv_begin &&
          it.kv_begin <= it.kv_end && it.kv_end <= T))
      bad = 1;
    // Every item holds a valid pair under these masks, as a pruned schedule
    // built from the same cu_seqlens does; an item that does not means the
    // device cu_seqlens differs from the one the schedule was built from.
    else if (!item_has_pair(cu, ndocs, it.q_begin, it.q_end, it.kv_begin, it.kv_end, causal))
      bad = 1;
    int h0, h1;
    item_heads_of(heads, i, Hq, h0, h1);
    const int nh = h1 - h0;
    // Whole key/value-head groups, or a piece inside one group.
    const bool whole = nh > 0 && nh % G == 0 && h0 % G == 0;
    const bool inside = nh > 0 && G % nh == 0 && h0 % nh == 0;
    if (!(0 <= h0 && h1 <= Hq && (whole || inside))) bad = 1;
    cnt += starts_group(i);
  }
  long long nseg_ll;
  long long off = block_exclusive_scan(cnt, scan_tmp, &nseg_ll);
  const int nseg = static_cast<int>(nseg_ll);
  for (int i = i0; i < i1; ++i)
    if (starts_group(i)) starts[off++] = i;
  if (tid == 0) starts[nseg] = n;
  __syncthreads();

  // Visit order: a group whose items are not all whole 128-key tiles long
  // (TASP pieces, for example) visits them by key start (ties in schedule
  // order), so that contiguous key ranges can be walked as one without a cut
  // tile at each seam. The order of the partial results a unit merges does
  // not change the result beyond rounding. Other groups, and groups of more
  // than 2048 items, keep the schedule order. One warp per group.
  {
    int32_t* order = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + L.off_order);
    const int wid = tid >> 5, lid = tid & 31;
    for (int sg = wid; sg < nseg; sg += 32) {
      const int g0 = starts[sg], g1 = starts[sg + 1];
      bool ragged = false;
      for (int i = g0 + lid; i < g1; i += 32)
        ragged |= ((__ldg(&items[i].kv_end) - __ldg(&items[i].kv_begin)) & 127) != 0;
      const bool sort = g1 - g0 <= 2048 && __any_sync(0xffffffffu, ragged);
      if (sort && lid == 0) any_sorted = 1;
      for (int i = g0 + lid; i < g1; i += 32) {
        int rank = i - g0;
        if (sort) {
          const int kb = __ldg(&items[i].kv_begin);
          rank = 0;
          for (int j = g0; j < g1; ++j) {
            const int kj = __ldg(&items[j].kv_begin);
            rank += (kj < kb) || (kj == kb && j < i);
          }
        }
        order[g0 + rank] = i;
      }
    }
  }
  for (int s = tid; s < nseg; s += 1024) {
    const int lo = starts[s], hi = starts[s + 1];
    const sp_item first = items[lo];
    long long tiles = 0;
    for (int i = lo; i < hi; ++i) tiles += (items[i].kv_end - items[i].kv_begin + 127) / 128;
    const int qg = (first.q_end - first.q_begin + rpu - 1) / rpu;
    SegEntry e;
    e.q_lo = first.q_begin;
    e.q_hi = first.q_end;
    e.item_lo = lo;
    e.item_hi = hi;
    e.unit_begin = 0;
    e.n_qgroups = qg;
    item_heads_of(heads, lo, Hq, e.h_lo, e.h_hi);
    tmp[s] = e;
    cost[s] = max(e.h_hi - e.h_lo, 0) > 0 ? tiles : 0;
  }
  __syncthreads();

  // Longest unit walk first (ties keep schedule order): the launch ends with
  // its last unit, so the units that walk the most keys start first (longest
  // processing time first list scheduling); inside a group the row groups run
  // last first, which under the causal mask is longest first too. Ordering by
  // a group's total work instead started a rank's short-document groups before
  // the tail of a long document, and the launch waited for those long units
  // at the end (1.2x the mean on one 128K-token packing's rank).
  if (tid == 0 && nseg > MAX_GROUPS) bad = 1;
  const bool sorted = nseg <= MAX_GROUPS;
  for (int s = tid; s < nseg; s += 1024) {
    int rank = s;
    if (sorted) {
      rank = 0;
      const long long cs = cost[s];
      for (int t2 = 0; t2 < nseg; ++t2) {
        const long long ct = cost[t2];
        rank += (ct > cs) || (ct == cs && t2 < s);
      }
    }
    segs[rank] = tmp[s];
  }
  __syncthreads();

  // The (Q range x head range) rectangles of different groups must not
  // overlap (each output row of each head is written by exactly one group).
  if (nseg <= MAX_GROUPS) {
    for (int s = tid; s < nseg; s += 1024) {
      const int a0 = segs[s].q_lo, a1 = segs[s].q_hi, g0 = segs[s].h_lo, g1 = segs[s].h_hi;
      for (int t2 = s + 1; t2 < nseg; ++t2)
        if (max(a0, segs[t2].q_lo) < min(a1, segs[t2].q_hi) &&
            max(g0, segs[t2].h_lo) < min(g1, segs[t2].h_hi))
          bad = 1;
    }
  }

  // Work-unit prefix over the sorted groups. With one query head per key/value
  // head (G = 1) and items over all heads, units run head by head across all
  // groups (each head's groups largest first), and the prefix is over one
  // head's units of each group. Group by group, the units running at once
  // would span about (number of SMs) / (row groups of a group) heads, each with
  // its own K/V: on the 64K-token 16-head layer that is ~300 MB against a
  // 129 MB L2, and the launch read 9.2 GB from DRAM (1.1 GB head by head). With
  // G > 1 the G heads of one K/V head are adjacent units already, and the
  // head-major order measured 0.6-1.5% slower on the GQA workloads.
  const bool kv_major = heads == nullptr && G == 1;
  const int schunk = (nseg + 1023) / 1024;
  const int s0 = min(nseg, tid * schunk), s1 = min(nseg, s0 + schunk);
  auto seg_units = [&](const SegEntry& e) {
    return static_cast<long long>(e.n_qgroups) * (kv_major ? G : (e.h_hi - e.h_lo));
  };
  long long units = 0;
  for (int s = s0; s < s1; ++s) units += seg_units(segs[s]);
  long long per_kv;
  long long ub = block_exclusive_scan(units, scan_tmp, &per_kv);
  for (int s = s0; s < s1; ++s) {
    segs[s].unit_begin = static_cast<int32_t>(ub);
    ub += seg_units(segs[s]);
  }
  const long long total = kv_major ? per_kv * Hkv : per_kv;
  __syncthreads();
  if (tid == 0) {
    const bool fail = bad || total > 0x7fffffffll;
    header[WS_N_SEGS] = fail ? 0 : nseg;
    header[WS_N_UNITS] = fail ? 0 : static_cast<int32_t>(total);
    header[WS_KV_UNITS] = (fail || !kv_major) ? 0 : static_cast<int32_t>(per_kv);
    header[WS_STATUS] = fail ? 1 : 0;
    header[WS_COUNTER] = 0;
    header[WS_ORDERED] = any_sorted;
    if (fail) atomicOr(err, ERR_INTERNAL_BIT);
  }
}

// Folds partial 2 into accumulator 1 in place, by the log-sum-exp rule. Each
// warp handles UNROLL (row, head) pairs per pass and issues every load of the
// pass (the LSE words and, for d <= 128, all of the O rows) before any of the
// arithmetic that needs them, so that enough bytes are in flight to keep HBM
// busy (the kernel is bandwidth bound: 12 bytes per O element). The merged LSE
// words are stored at the end of the pass, after every lane has read them.
constexpr int MERGE_UNROLL = 4;

__global__ void __launch_bounds__(256)
lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                 const float* __restrict__ o_part, const float* __restrict__ lse_part, int rows,
                 int Hq, int d) {
  const int lane = threadIdx.x & 31;
  const long long n = static_cast<long long>(rows) * Hq;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5) * MERGE_UNROLL;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int nv = d >> 2;  // float4 per O row
  for (long long w0 = (static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * MERGE_UNROLL;
       w0 < n; w0 += wstride) {
    size_t li[MERGE_UNROLL];
    float l1[MERGE_UNROLL], l2[MERGE_UNROLL];
#pragma unroll
    for (int k = 0; k < MERGE_UNROLL; ++k) {
      const long long w = w0 + k;
      l1[k] = l2[k] = NEG_INF;
      li[k] = 0;
      if (w >= n) continue;
      const int row = static_cast<int>(w / Hq), h = static_cast<int>(w % Hq);
      li[k] = static_cast<size_t>(h) * rows + row;
      l1[k] = lse_acc[li[k]];
      l2[k] = __ldg(lse_part + li[k]);
    }
    // The first float4 column of every O row (the only one when d <= 128).
    float4 x[MERGE_UNROLL], y[MERGE_UNROLL];
    if (lane < nv) {
#pragma unroll
      for (int k = 0; k < MERGE_UNROLL; ++k) {
        if (w0 + k >= n) continue;
        x[k] = reinterpret_cast<const float4*>(o_acc + static_cast<size_t>(w0 + k) * d)[lane];
        y[k] = __ldg(reinterpret_cast<const float4*>(o_part + static_cast<size_t>(w0 + k) * d) + lane);
      }
    }
    // Weights of the UNROLL pairs.
    float w1[MERGE_UNROLL], w2[MERGE_UNROLL], L[MERGE_UNROLL];
#pragma unroll
    for (int k = 0; k < MERGE_UNROLL; ++k) {
      const float M = fmaxf(l1[k], l2[k]);
      w1[k] = w2[k] = 0.f;
      L[k] = NEG_INF;
      if (M != NEG_INF) {
        const float e1 = expf(l1[k] - M), e2 = expf(l2[k] - M);
        const float s = e1 + e2;
        L[k] = M + logf(s);
        const float inv = 1.f / s;
        w1[k] = e1 * inv;
        w2[k] = e2 * inv;
      }
    }
    for (int c = lane; c < nv; c += 32) {
      if (c != lane) {
#pragma unroll
        for (int k = 0; k < MERGE_UNROLL; ++k) {
          if (w0 + k >= n) continue;
          x[k] = reinterpret_cast<const float4*>(o_acc + static_cast<size_t>(w0 + k) * d)[c];
          y[k] = __ldg(reinterpret_cast<const float4*>(o_part + static_cast<size_t>(w0 + k) * d) + c);
        }
      }
#pragma unroll
      for (int k = 0; k < MERGE_UNROLL; ++k) {
        if (w0 + k >= n) continue;
        reinterpret_cast<float4*>(o_acc + static_cast<size_t>(w0 + k) * d)[c] =
            make_float4(w1[k] * x[k].x + w2[k] * y[k].x, w1[k] * x[k].y + w2[k] * y[k].y,
                        w1[k] * x[k].z + w2[k] * y[k].z, w1[k] * x[k].w + w2[k] * y[k].w);
      }
    }
    // Every lane has read the accumulator's LSE words of this pass.
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < MERGE_UNROLL; ++k)
        if (w0 + k < n) lse_acc[li[k]] = L[k];
    }
  }
}

__global__ void wait_selftest_kernel(unsigned long long timeout_ns, unsigned* err) {
  __shared__ __align__(8) unsigned long long barmem;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(&barmem);
    abort_flag = 0;
    mbar_init(bar, 1);
    mbar_fence_init();
    // Nothing ever arrives on bar: the wait must give up on its own.
    mbar_wait_bounded(bar, 0, timeout_ns, err, &abort_flag);
  }
}

}  // namespace

cudaError_t launch_prep(const sp_item* items, const int32_t* item_heads, int64_t n_items, int32_t T,
                        int32_t Hq, int32_t Hkv, int32_t rows_per_unit, void* workspace, unsigned* err,
                        const int32_t* cu, int32_t ndocs, int32_t causal, cudaStream_t st) {
  prep_kernel<<<1, 1024, 0, st>>>(items, item_heads, static_cast<int>(n_items), T, Hq, Hkv, rows_per_unit,
                                  static_cast<int32_t*>(workspace), err, cu, ndocs, causal ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                             int32_t rows, int32_t Hq, int32_t d, int grid, cudaStream_t st) {
  lse_merge_kernel<<<grid, 256, 0, st>>>(o_acc, lse_acc, o_part, lse_part, rows, Hq, d);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned long long timeout_ns, unsigned* err, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns, err);
  return cudaGetLastError();
}

}  // namespace sp
