// Internal declarations shared by the translation units of libsp_attn.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/sp_attn.h"

namespace sp {

// Devices a process may use the library on (per-device state is kept in
// arrays of this size; larger device ids are rejected).
constexpr int MAX_DEVICES = 64;

// Error bits recorded in the per-device error word.
enum : unsigned { ERR_TIMEOUT_BIT = 1u, ERR_INTERNAL_BIT = 2u };

// One group of items that share a rank, a Q range and a range of query
// heads. After the set-up kernel the table is sorted by estimated cost,
// largest first.
struct SegEntry {
  int32_t q_lo, q_hi;        // Q rows of the group
  int32_t item_lo, item_hi;  // items [item_lo, item_hi) in schedule order
  int32_t unit_begin;        // first work unit of the group
  int32_t n_qgroups;         // row groups of rows_per_unit rows
  int32_t h_lo, h_hi;        // query heads [h_lo, h_hi) (all heads unless a head split is given)
};
static_assert(sizeof(SegEntry) == 32, "SegEntry is 32 bytes");

// Workspace header (int32 words).
// WS_COUNTER: next work unit to hand out (reset to 0 by the set-up kernel).
// WS_BWD_COUNTER: the backward dK/dV kernel's unit queue.
// WS_ORDERED: nonzero when some group's items are visited in key order (the
// set-up kernel's visit order) rather than schedule order.
// WS_KV_UNITS: units per key/value head when units run key/value-head-major
// across all groups (Hq == Hkv and every item covers all heads); 0 when they
// run group by group.
enum : int { WS_N_SEGS = 0, WS_N_UNITS = 1, WS_STATUS = 2, WS_COUNTER = 3, WS_BWD_COUNTER = 4,
             WS_ORDERED = 5, WS_KV_UNITS = 6, WS_HEADER_WORDS = 16 };

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const int32_t* cu;
  int32_t ndocs;
  int32_t T, Hq, Hkv, d;
  int32_t causal;
  float scale;       // multiplies q.k
  float scale_log2;  // scale * log2(e)
  // Work description: either a device table produced by the set-up kernel
  // (header != nullptr) or one inline group holding one inline item.
  const sp_item* items;
  const int32_t* item_order;  // visit order of the items (nullptr: schedule order)
  const SegEntry* segs;
  const int32_t* header;
  int32_t* work_counter;  // dynamic unit queue (nullptr: static striding over CTAs)
  sp_item inline_item;
  SegEntry inline_seg;
  int32_t inline_n_units;
  int32_t rows_per_unit;
  // Output: mode 0 writes O [T][Hq][d] (bf16 or fp32) and LSE [Hq][T];
  // mode 1 writes fp32 O [t - row_base][Hq][d] and LSE [Hq][n_rows].
  int32_t out_mode;
  int32_t row_base, n_rows;
  unsigned* err;
  unsigned long long timeout_ns;
};

// Arguments of the backward kernels. fwd holds the forward's inputs, shapes
// and schedule tables (its o and lse fields are unused).
struct BwdArgs {
  AttnArgs fwd;
  const float* lse;    // [Hq][T] natural-log LSE written by the forward
  const float* ndsc;   // [Hq][T] -scale * D_i, D_i = dO_i . O_i
  const float* nlse2;  // [Hq][T] -LSE_i * log2(e)
  int32_t* unit_counter;  // fused kernel's work-unit queue (zeroed by the row-dot kernel)
  float* dqacc;       // fp32 [T][Hq][d] dQ accumulator (zeroed by the row-dot kernel)
  int32_t* status;    // nonzero when the row-dot kernel found cu_seqlens invalid (nothing is written)
  void* dq;           // bf16 [T][Hq][d]
  void* dk;           // bf16 [T][Hkv][d]
  void* dv;           // bf16 [T][Hkv][d]
};

// Launchers (return cudaGetLastError() of the launch).
// item_heads: NULL (every item covers all Hq heads) or int32 [n][2] query-head
// ranges; a range must cover whole key/value-head groups or lie inside one.
cudaError_t launch_prep(const sp_item* items, const int32_t* item_heads, int64_t n_items, int32_t T,
                        int32_t Hq, int32_t Hkv, int32_t rows_per_unit, void* workspace, unsigned* err,
                        const int32_t* cu, int32_t ndocs, int32_t causal, cudaStream_t st);
cudaError_t launch_attn_simt(const AttnArgs& a, int grid, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnArgs& a, const void* tmap_q, const void* tmap_k,
                           const void* tmap_v, int grid, cudaStream_t st);
// CTA-pair variant (d = 128, Hq / Hkv even, every item over all heads): tmap_k64
// has a 64-row box. Units 2v and 2v+1 (two query heads of one key/value head,
// same rows) run on the two CTAs of cluster-pair unit v.
cudaError_t launch_attn_tc_pair(const AttnArgs& a, const void* tmap_q, const void* tmap_k64,
                                const void* tmap_v, int n_pairs_hint, cudaStream_t st);
cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                             int32_t rows, int32_t Hq, int32_t d, int grid, cudaStream_t st);
cudaError_t launch_bwd_rowdot(const void* o, const void* dout, const float* lse, float* ndsc, float* nlse2,
                              float* dqacc, int32_t* unit_counter, int32_t* status, const int32_t* cu,
                              int ndocs, unsigned* err, int T, int Hq, int d, float scale, int grid,
                              cudaStream_t st);
// The fused dK/dV/dQ kernel (key/value tiles stationary, dQ reduced into
// dqacc), then dQ rounded from dqacc to bf16.
cudaError_t launch_bwd_tc(const BwdArgs& a, const void* tmap_q, const void* tmap_k,
                          const void* tmap_v, const void* tmap_do, int grid, cudaStream_t st);
cudaError_t launch_wait_selftest(unsigned long long timeout_ns, unsigned* err, cudaStream_t st);

// Rows per work unit of each kernel.
constexpr int TC_ROWS_PER_UNIT = 256;
constexpr int SIMT_ROWS_PER_UNIT = 128;
constexpr int BWD_ROWS_PER_UNIT = 128;

}  // namespace sp
