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

// ---------------------------------------------------------------------------
// Unit records: what every role of a forward kernel needs to run a unit,
// built once by a scheduler warp and passed through shared memory, so that
// the table searches (unit decode, the Q tiles' documents) and the walk over
// the items to the unit's first tile stay off the other roles' path. Words:
// the unit (< 0: no more work), its query head and first row, the two Q tiles
// (bounds, documents), and the cursor standing on the first tile (a reader's
// first next_tile returns that tile without reading an item).
constexpr int UREC_WORDS = 32;  // slot stride (int32 words)
enum { UR_V = 0, UR_H = 1, UR_Q0 = 2, UR_QT = 3, UR_CUR = 13, UR_N = 19 };

__device__ __forceinline__ void build_unit_record(const AttnArgs& a, int unit, int v, int (&w)[UR_N]) {
  const UnitInfo ui = unit_info(a, unit);
  const QTile qt[2] = {make_qtile(a, ui, 0), make_qtile(a, ui, 1)};
  Cursor cur = make_cursor(a, ui, qt, a.causal);
  int ka = 0, kb = 0, cls[2];
  if (next_tile(a, cur, qt, ka, kb, cls)) cur.k0 = ka;  // back onto the first tile
  w[UR_V] = v;
  w[UR_H] = ui.h;
  w[UR_Q0] = ui.q0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    w[UR_QT + 5 * i + 0] = qt[i].qa;
    w[UR_QT + 5 * i + 1] = qt[i].qb;
    w[UR_QT + 5 * i + 2] = qt[i].ds;
    w[UR_QT + 5 * i + 3] = qt[i].de;
    w[UR_QT + 5 * i + 4] = qt[i].one_doc;
  }
  w[UR_CUR + 0] = cur.item;
  w[UR_CUR + 1] = cur.item_end;
  w[UR_CUR + 2] = cur.kv_e;
  w[UR_CUR + 3] = cur.k0;
  w[UR_CUR + 4] = cur.lo;
  w[UR_CUR + 5] = cur.hi;
}

// Reads a record (unit >= 0); dh is added to the recorded query head.
__device__ __forceinline__ void read_unit_record(const volatile int* rs, int dh, int& h, int& q0,
                                                 QTile (&qt)[2], Cursor& cur) {
  h = rs[UR_H] + dh;
  q0 = rs[UR_Q0];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    qt[i].qa = rs[UR_QT + 5 * i + 0];
    qt[i].qb = rs[UR_QT + 5 * i + 1];
    qt[i].ds = rs[UR_QT + 5 * i + 2];
    qt[i].de = rs[UR_QT + 5 * i + 3];
    qt[i].one_doc = rs[UR_QT + 5 * i + 4];
  }
  cur.item = rs[UR_CUR + 0];
  cur.item_end = rs[UR_CUR + 1];
  cur.kv_e = rs[UR_CUR + 2];
  cur.k0 = rs[UR_CUR + 3];
  cur.lo = rs[UR_CUR + 4];
  cur.hi = rs[UR_CUR + 5];
}

}  // namespace sp
