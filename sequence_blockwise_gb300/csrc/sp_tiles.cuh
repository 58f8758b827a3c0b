// Tile walk shared by the attention kernels: the Q tiles of a work unit, the
// classification of a (Q tile, key tile) pair, and the cursor over a unit's
// items (key ranges clipped to the keys some row of the unit may attend).
#pragma once

#include "sp_device.cuh"

namespace sp {

constexpr int CLS_SKIP = 0, CLS_MASKED = 1, CLS_FULL = 2;

struct QTile {
  int qa, qb;   // valid rows [qa, qb) (empty when qa >= qb)
  int ds, de;   // document start of row qa, document end of row qb-1
  int one_doc;  // rows all in one document
};

__device__ __forceinline__ QTile make_qtile(const AttnArgs& a, const UnitInfo& ui, int i) {
  QTile t;
  t.qa = ui.q0 + 128 * i;
  t.qb = min(t.qa + 128, ui.q_hi);
  if (t.qb <= t.qa) {
    t.qa = t.qb = 0;
    t.ds = t.de = 0;
    t.one_doc = 0;
    return t;
  }
  const int d0 = doc_of(a.cu, a.ndocs, t.qa);
  const int d1 = doc_of(a.cu, a.ndocs, t.qb - 1);
  t.ds = __ldg(a.cu + d0);
  t.de = __ldg(a.cu + d1 + 1);
  t.one_doc = (d0 == d1);
  return t;
}

__device__ __forceinline__ int classify(const QTile& t, int ka, int kb, int causal) {
  if (t.qa >= t.qb) return CLS_SKIP;
  if (causal && ka > t.qb - 1) return CLS_SKIP;
  if (t.de <= ka || kb <= t.ds) return CLS_SKIP;
  if (t.qb - t.qa == 128 && kb - ka == 128 && t.one_doc && ka >= t.ds && kb <= t.de &&
      (!causal || kb - 1 <= t.qa))
    return CLS_FULL;
  return CLS_MASKED;
}

// item_end holds the end of the unit's items in its low 30 bits and, in bit
// 30, whether the items are visited in the set-up kernel's key order (so that
// the flag costs no register on the per-tile path).
constexpr int CUR_ORDERED = 1 << 30, CUR_END_MASK = CUR_ORDERED - 1;

struct Cursor {
  int item, item_end, kv_e, k0;
  int lo, hi;  // keys any row of the unit may attend: [lo, hi)
};

// Cursor over a unit's items. Each item's key range is first clipped to the
// keys some row of the unit may attend (the documents of its rows, and keys
// up to its last row when causal), so that no tile is visited for keys that
// are masked for every row; tiles start at the clipped start.
__device__ __forceinline__ Cursor make_cursor(const AttnArgs& a, const UnitInfo& ui, const QTile (&qt)[2],
                                              int causal) {
  const bool ordered = a.header && a.item_order && __ldg(a.header + WS_ORDERED);
  Cursor c{ui.item_lo, ui.item_hi | (ordered ? CUR_ORDERED : 0), 0, 0, 0, 0};
  const bool e0 = qt[0].qa < qt[0].qb, e1 = qt[1].qa < qt[1].qb;
  if (!e0 && !e1) {
    c.item = ui.item_hi;  // no valid row: no tile
    return c;
  }
  c.lo = e0 ? qt[0].ds : qt[1].ds;
  c.hi = e1 ? qt[1].de : qt[0].de;
  if (causal) c.hi = min(c.hi, (e1 ? qt[1].qb : qt[0].qb));
  return c;
}

// Advances to the next 128-key tile of the unit that is not SKIP for both Q
// tiles. Every role runs this same function, so all agree on the sequence.
// When the set-up kernel reordered some group (header word WS_ORDERED, read
// once per unit by make_cursor), items are visited in its key order, and
// items whose clipped key ranges follow one another without a gap are walked
// as one range, so that no tile is cut at the seam (TASP pieces of one chunk,
// for example); otherwise items are walked in schedule order.
__device__ __forceinline__ bool next_tile(const AttnArgs& a, Cursor& c, const QTile (&qt)[2],
                                          int& ka, int& kb, int (&cls)[2]) {
  while (true) {
    if (c.k0 >= c.kv_e) {
      const int end = c.item_end & CUR_END_MASK;
      if (c.item >= end) return false;
      const int32_t* order = (c.item_end & CUR_ORDERED) ? a.item_order : nullptr;
      int b, e;
      item_range(a, c.item, b, e, order);
      ++c.item;
      c.k0 = max(b, c.lo);
      c.kv_e = min(e, c.hi);
      while (order && c.k0 < c.kv_e && c.item < end) {
        item_range(a, c.item, b, e, order);
        const int nb = max(b, c.lo), ne = min(e, c.hi);
        if (nb != c.kv_e || ne <= nb) break;
        c.kv_e = ne;
        ++c.item;
      }
      continue;
    }
    ka = c.k0;
    kb = min(c.k0 + 128, c.kv_e);
    c.k0 += 128;
    cls[0] = classify(qt[0], ka, kb, a.causal);
    cls[1] = classify(qt[1], ka, kb, a.causal);
    if (cls[0] != CLS_SKIP || cls[1] != CLS_SKIP) return true;
  }
}

}  // namespace sp
