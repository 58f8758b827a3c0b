// Layout of the caller-provided workspace of sp_packed_attention:
// [header: 16 int32][sorted groups][unsorted groups][group starts][group costs]
// [item visit order].
#pragma once

#include <cstddef>

#include "sp_internal.h"

namespace sp {

struct WsLayout {
  size_t off_segs, off_tmp, off_starts, off_cost, off_order, total;
};

__host__ __device__ inline WsLayout ws_layout(long long n) {
  WsLayout L;
  size_t o = WS_HEADER_WORDS * sizeof(int32_t);
  L.off_segs = o;
  o += static_cast<size_t>(n) * sizeof(SegEntry);
  L.off_tmp = o;
  o += static_cast<size_t>(n) * sizeof(SegEntry);
  L.off_starts = o;
  o += (static_cast<size_t>(n) + 1) * sizeof(int32_t);
  o = (o + 15) & ~static_cast<size_t>(15);
  L.off_cost = o;
  o += static_cast<size_t>(n) * sizeof(long long);
  L.off_order = o;
  o += static_cast<size_t>(n) * sizeof(int32_t);
  L.total = (o + 255) & ~static_cast<size_t>(255);
  return L;
}

}  // namespace sp
