// C-ABI entry points of libsp_attn: argument checks, TMA descriptors, and
// launches. The arithmetic is in the kernels; this file only validates and
// dispatches.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "sp_internal.h"
#include "sp_workspace.h"

// Per-device error word (each device holds its own copy of module globals).
__device__ unsigned g_sp_error;

namespace {

using sp::AttnArgs;

constexpr int kMaxDevices = sp::MAX_DEVICES;
constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;  // 4 s of GPU time per wait

std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

sp_status cuda_fail(cudaError_t e) { return e == cudaSuccess ? SP_OK : SP_ERR_CUDA; }

bool device_state(unsigned** err, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sp_error) != cudaSuccess) return false;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
    g_sms[dev] = n;
  }
  *err = g_err_ptr[dev];
  *sms = g_sms[dev];
  return true;
}

bool encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Rank-3 bf16 map over [T][H][d] with a {64, 1, box_rows} box and 128-byte
// swizzle: one load brings box_rows tokens x 64 dims of one head, laid out as
// the tensor core reads a K-major (Q, K) or MN-major (V) operand.
bool encode_map(CUtensorMap* m, const void* base, int T, int H, int d, int box_rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

unsigned long long timeout_ns() {
  static unsigned long long v = [] {
    const char* s = std::getenv("SP_ATTN_WAIT_TIMEOUT_NS");
    if (s && *s) {
      const unsigned long long x = std::strtoull(s, nullptr, 10);
      if (x > 0) return x;
    }
    return kDefaultTimeoutNs;
  }();
  return v;
}

// Shared shape checks of the attention entry points.
sp_status check_shapes(int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype, int32_t ndocs,
                       float scale) {
  if (T < 0 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0) return SP_ERR_INVALID_ARG;
  if (dtype != SP_DTYPE_BF16 && dtype != SP_DTYPE_FP32) return SP_ERR_INVALID_ARG;
  if (T > 0 && ndocs < 1) return SP_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return SP_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SP_ERR_UNSUPPORTED;
  return SP_OK;
}

AttnArgs base_args(const void* q, const void* k, const void* v, void* o, float* lse, int32_t T,
                   int32_t Hq, int32_t Hkv, int32_t d, const int32_t* cu, int32_t ndocs,
                   int32_t causal, float scale, unsigned* err) {
  AttnArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.cu = cu;
  a.ndocs = ndocs;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.err = err;
  a.timeout_ns = timeout_ns();
  return a;
}

// heads_full: every item covers all query heads, so units come in pairs of
// query heads sharing a key/value head whenever Hq / Hkv is even.
sp_status launch_attention(AttnArgs& a, sp_dtype dtype, int sms, cudaStream_t st, int n_units_hint,
                           bool heads_full) {
  if (dtype == SP_DTYPE_BF16) {
    if (!encoder()) return SP_ERR_CUDA;
    CUtensorMap mq, mk, mv;
    if (heads_full && a.d == 128 && (a.Hq / a.Hkv) % 2 == 0) {
      // CTA pairs: each CTA loads 64 keys of a K tile and 64 dims of a V tile.
      if (!encode_map(&mq, a.q, a.T, a.Hq, a.d) || !encode_map(&mk, a.k, a.T, a.Hkv, a.d, 64) ||
          !encode_map(&mv, a.v, a.T, a.Hkv, a.d))
        return SP_ERR_CUDA;
      return cuda_fail(sp::launch_attn_tc_pair(a, &mq, &mk, &mv, n_units_hint / 2, st));
    }
    if (!encode_map(&mq, a.q, a.T, a.Hq, a.d) || !encode_map(&mk, a.k, a.T, a.Hkv, a.d) ||
        !encode_map(&mv, a.v, a.T, a.Hkv, a.d))
      return SP_ERR_CUDA;
    int grid = sms;
    if (n_units_hint > 0 && n_units_hint < grid) grid = n_units_hint;
    return cuda_fail(sp::launch_attn_tc(a, &mq, &mk, &mv, grid, st));
  }
  int grid = sms * 4;
  if (n_units_hint > 0 && n_units_hint < grid) grid = n_units_hint;
  return cuda_fail(sp::launch_attn_simt(a, grid, st));
}

}  // namespace

extern "C" {

sp_status sp_partial_attn(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                          int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                          int32_t q_begin, int32_t q_end, int32_t kv_begin, int32_t kv_end,
                          const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal, float scale,
                          void* stream) {
  sp_status s = check_shapes(T, Hq, Hkv, d, dtype, ndocs, scale);
  if (s != SP_OK) return s;
  if (q_begin < 0 || q_end < q_begin || q_end > T || kv_begin < 0 || kv_end < kv_begin || kv_end > T)
    return SP_ERR_INVALID_ARG;
  if (q_begin == q_end) return SP_OK;
  if (!q || !k || !v || !o_part || !lse_part || !cu_seqlens_dev) return SP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part)) return SP_ERR_INVALID_ARG;
  unsigned* err;
  int sms;
  if (!device_state(&err, &sms)) return SP_ERR_CUDA;
  AttnArgs a = base_args(q, k, v, o_part, lse_part, T, Hq, Hkv, d, cu_seqlens_dev, ndocs, causal,
                         scale, err);
  const int rpu = dtype == SP_DTYPE_BF16 ? sp::TC_ROWS_PER_UNIT : sp::SIMT_ROWS_PER_UNIT;
  const int rows = q_end - q_begin;
  const int qg = (rows + rpu - 1) / rpu;
  a.items = nullptr;
  a.segs = nullptr;
  a.header = nullptr;
  a.inline_item = sp_item{0, 0, 0, q_begin, q_end, kv_begin, kv_end, 0};
  a.inline_seg = sp::SegEntry{q_begin, q_end, 0, 1, 0, qg, 0, Hq};
  a.inline_n_units = qg * Hq;
  a.rows_per_unit = rpu;
  a.out_mode = 1;
  a.row_base = q_begin;
  a.n_rows = rows;
  return launch_attention(a, dtype, sms, static_cast<cudaStream_t>(stream), a.inline_n_units, true);
}

sp_status sp_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                       int32_t rows, int32_t Hq, int32_t d, void* stream) {
  if (rows < 0 || Hq < 1 || d < 4 || d % 4 != 0) return SP_ERR_INVALID_ARG;
  if (rows == 0) return SP_OK;
  if (!o_acc || !lse_acc || !o_part || !lse_part) return SP_ERR_INVALID_ARG;
  if (!aligned16(o_acc) || !aligned16(o_part)) return SP_ERR_INVALID_ARG;
  unsigned* err;
  int sms;
  if (!device_state(&err, &sms)) return SP_ERR_CUDA;
  const long long warps = (static_cast<long long>(rows) * Hq + 3) / 4;  // 4 (row, head) pairs per warp pass
  long long grid = (warps + 7) / 8;
  // Many short blocks (16 waves of the 3 resident per SM, a few grid-stride
  // passes each) balance the SMs' finishing times: on the 64K-row, 16-head
  // partials, 0.253 ms against 0.286 with 16 blocks per SM, 0.260 uncapped and
  // 0.298 with a single wave.
  if (grid > static_cast<long long>(sms) * 48) grid = static_cast<long long>(sms) * 48;
  return cuda_fail(sp::launch_lse_merge(o_acc, lse_acc, o_part, lse_part, rows, Hq, d,
                                        static_cast<int>(grid), static_cast<cudaStream_t>(stream)));
}

size_t sp_packed_attention_workspace_size(int64_t n_items) {
  if (n_items < 0) n_items = 0;
  return sp::ws_layout(n_items).total;
}

sp_status sp_packed_attention(const void* q, const void* k, const void* v, void* o, float* lse,
                              int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                              const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal, float scale,
                              const sp_item* items_dev, int64_t n_items, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return sp_packed_attention_ex(q, k, v, o, lse, T, Hq, Hkv, d, dtype, cu_seqlens_dev, ndocs, causal,
                                scale, items_dev, nullptr, n_items, workspace, workspace_bytes, stream);
}

sp_status sp_packed_attention_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                                 const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal,
                                 float scale, const sp_item* items_dev, const int32_t* item_heads_dev,
                                 int64_t n_items, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  sp_status s = check_shapes(T, Hq, Hkv, d, dtype, ndocs, scale);
  if (s != SP_OK) return s;
  if (n_items < 0 || n_items >= (1ll << 30)) return SP_ERR_INVALID_ARG;
  if (T == 0 || n_items == 0) return SP_OK;
  if (!q || !k || !v || !o || !lse || !cu_seqlens_dev || !items_dev || !workspace)
    return SP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(items_dev) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(item_heads_dev) & 7u) != 0)
    return SP_ERR_INVALID_ARG;
  if (workspace_bytes < sp_packed_attention_workspace_size(n_items)) return SP_ERR_BUFFER_TOO_SMALL;
  unsigned* err;
  int sms;
  if (!device_state(&err, &sms)) return SP_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rpu = dtype == SP_DTYPE_BF16 ? sp::TC_ROWS_PER_UNIT : sp::SIMT_ROWS_PER_UNIT;
  cudaError_t e = sp::launch_prep(items_dev, item_heads_dev, n_items, T, Hq, Hkv, rpu, workspace, err,
                                  cu_seqlens_dev, ndocs, causal, st);
  if (e != cudaSuccess) return SP_ERR_CUDA;
  AttnArgs a = base_args(q, k, v, o, lse, T, Hq, Hkv, d, cu_seqlens_dev, ndocs, causal, scale, err);
  const sp::WsLayout L = sp::ws_layout(n_items);
  a.items = items_dev;
  a.item_order = reinterpret_cast<const int32_t*>(static_cast<const char*>(workspace) + L.off_order);
  a.header = static_cast<const int32_t*>(workspace);
  a.work_counter = static_cast<int32_t*>(workspace) + sp::WS_COUNTER;
  a.segs = reinterpret_cast<const sp::SegEntry*>(static_cast<const char*>(workspace) + L.off_segs);
  a.rows_per_unit = rpu;
  a.out_mode = 0;
  a.row_base = 0;
  a.n_rows = T;
  return launch_attention(a, dtype, sms, st, 0, item_heads_dev == nullptr);
}

}  // extern "C"

namespace {

// Backward workspace: [header (the unit counter)][-scale D][-LSE log2 e]
// [fp32 dQ accumulator]; each part 256-byte aligned. The accumulator is sized
// for d = 128, the largest head dimension.
struct BwdWs {
  size_t off_ndsc, off_nlse2, off_dqacc, total;
};

BwdWs bwd_ws(int32_t T, int32_t Hq) {
  auto r256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t rows = static_cast<size_t>(T) * static_cast<size_t>(Hq);
  BwdWs L;
  L.off_ndsc = r256(sp::WS_HEADER_WORDS * sizeof(int32_t));
  L.off_nlse2 = L.off_ndsc + r256(rows * sizeof(float));
  L.off_dqacc = L.off_nlse2 + r256(rows * sizeof(float));
  L.total = L.off_dqacc + r256(rows * 128 * sizeof(float));
  return L;
}

}  // namespace

extern "C" {

size_t sp_packed_attention_backward_workspace_size(int64_t n_items, int32_t T, int32_t Hq) {
  (void)n_items;
  if (T < 0) T = 0;
  if (Hq < 0) Hq = 0;
  return bwd_ws(T, Hq).total;
}

sp_status sp_packed_attention_backward(const void* q, const void* k, const void* v, const void* o,
                                       const void* dout, const float* lse, void* dq, void* dk,
                                       void* dv, int32_t T, int32_t Hq, int32_t Hkv, int32_t d,
                                       sp_dtype dtype, const int32_t* cu_seqlens_dev, int32_t ndocs,
                                       int32_t causal, float scale, const sp_item* items_dev,
                                       int64_t n_items, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  sp_status s = check_shapes(T, Hq, Hkv, d, dtype, ndocs, scale);
  if (s != SP_OK) return s;
  if (dtype != SP_DTYPE_BF16) return SP_ERR_UNSUPPORTED;
  if (n_items < 0 || n_items >= (1ll << 30)) return SP_ERR_INVALID_ARG;
  if (T == 0) return SP_OK;
  if (n_items == 0) return SP_ERR_INVALID_ARG;  // a complete schedule has items whenever T > 0
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !cu_seqlens_dev || !items_dev ||
      !workspace)
    return SP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(items_dev) ||
      !aligned16(workspace))
    return SP_ERR_INVALID_ARG;
  if (workspace_bytes < sp_packed_attention_backward_workspace_size(n_items, T, Hq))
    return SP_ERR_BUFFER_TOO_SMALL;
  unsigned* err;
  int sms;
  if (!device_state(&err, &sms)) return SP_ERR_CUDA;
  if (!encoder()) return SP_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const BwdWs L = bwd_ws(T, Hq);
  char* ws = static_cast<char*>(workspace);
  float* ndsc = reinterpret_cast<float*>(ws + L.off_ndsc);
  float* nlse2 = reinterpret_cast<float*>(ws + L.off_nlse2);
  float* dqacc = reinterpret_cast<float*>(ws + L.off_dqacc);
  int32_t* unit_counter = reinterpret_cast<int32_t*>(ws) + sp::WS_BWD_COUNTER;
  int32_t* status = reinterpret_cast<int32_t*>(ws) + sp::WS_STATUS;

  const long long warps = static_cast<long long>(T) * Hq;
  long long g = (warps + 7) / 8;
  if (g > static_cast<long long>(sms) * 16) g = static_cast<long long>(sms) * 16;
  cudaError_t e = sp::launch_bwd_rowdot(o, dout, lse, ndsc, nlse2, dqacc, unit_counter, status,
                                        cu_seqlens_dev, ndocs, err, T, Hq, d, scale, static_cast<int>(g), st);
  if (e != cudaSuccess) return SP_ERR_CUDA;

  sp::BwdArgs b;
  std::memset(&b, 0, sizeof b);
  b.fwd = base_args(q, k, v, nullptr, nullptr, T, Hq, Hkv, d, cu_seqlens_dev, ndocs, causal, scale, err);
  b.lse = lse;
  b.ndsc = ndsc;
  b.nlse2 = nlse2;
  b.unit_counter = unit_counter;
  b.dqacc = dqacc;
  b.status = status;
  b.dq = dq;
  b.dk = dk;
  b.dv = dv;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_map(&mq, q, T, Hq, d, 64) || !encode_map(&mk, k, T, Hkv, d, 64) ||
      !encode_map(&mv, v, T, Hkv, d, 64) || !encode_map(&mdo, dout, T, Hq, d, 64))
    return SP_ERR_CUDA;
  return cuda_fail(sp::launch_bwd_tc(b, &mq, &mk, &mv, &mdo, sms, st));
}

sp_status sp_check_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return SP_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_sp_error, sizeof v) != cudaSuccess) return SP_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_sp_error, &zero, sizeof zero) != cudaSuccess) return SP_ERR_CUDA;
  }
  if (v & sp::ERR_TIMEOUT_BIT) return SP_ERR_TIMEOUT;
  if (v & sp::ERR_INTERNAL_BIT) return SP_ERR_INTERNAL;
  return SP_OK;
}

sp_status sp_selftest_bounded_wait(uint64_t timeout_ns_arg, void* stream) {
  unsigned* err;
  int sms;
  if (!device_state(&err, &sms)) return SP_ERR_CUDA;
  return cuda_fail(sp::launch_wait_selftest(timeout_ns_arg, err, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the workspace is a fixed array in this module.

namespace {

// Scratch shared by every sp_packed_attention_static_ws call on a device. Host
// code must not use the symbol itself as a pointer (it names a host-side
// stand-in); it uses the device address looked up once per device below.
static __device__ __align__(256) unsigned char g_static_ws[SP_STATIC_WS_BYTES];

std::mutex g_static_mu;
void* g_static_ws_dev[kMaxDevices] = {};

}  // namespace

extern "C" sp_status sp_packed_attention_static_ws(const void* q, const void* k, const void* v, void* o,
                                                   float* lse, int32_t T, int32_t Hq, int32_t Hkv,
                                                   int32_t d, sp_dtype dtype,
                                                   const int32_t* cu_seqlens_dev, int32_t ndocs,
                                                   int32_t causal, float scale,
                                                   const sp_item* items_dev, int64_t n_items,
                                                   void* stream) {
  // Argument errors are returned before any CUDA call, as by sp_packed_attention.
  const sp_status s = check_shapes(T, Hq, Hkv, d, dtype, ndocs, scale);
  if (s != SP_OK) return s;
  if (n_items < 0) return SP_ERR_INVALID_ARG;
  if (n_items > SP_STATIC_WS_MAX_ITEMS ||
      sp_packed_attention_workspace_size(n_items) > SP_STATIC_WS_BYTES)
    return SP_ERR_BUFFER_TOO_SMALL;
  if (T == 0 || n_items == 0) return SP_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SP_ERR_CUDA;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ws_dev[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return SP_ERR_CUDA;
      g_static_ws_dev[dev] = p;
    }
    ws = g_static_ws_dev[dev];
  }
  return sp_packed_attention(q, k, v, o, lse, T, Hq, Hkv, d, dtype, cu_seqlens_dev, ndocs, causal,
                             scale, items_dev, n_items, ws, SP_STATIC_WS_BYTES, stream);
}
