// Plain fp64 CPU oracle for blockwise packed attention and its chunk schedules.
//
// TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the CPU
// baseline leg of the benchmark may load this code. The product library never
// links, includes or calls it, and this file includes nothing from the product.
//
// What it computes (sources):
//  * Exact softmax attention restricted to each packed document, optionally
//    causal. HSAP abstract ("correctly compute causal attention on the
//    hybrid-context packed sequences"; packing causes "cross-contamination"),
//    TASP abstract ("enable each Q tensor to access all KV tensors"). The
//    formula is the textbook one: s_j = <q_i, k_j> * scale over the valid key
//    set V(i) = { j : doc(j) == doc(i) and (not causal or j <= i) },
//    LSE = log sum_j exp(s_j), O = sum_j exp(s_j - LSE) v_j.
//  * GQA: query head h reads key/value head h / (Hq / Hkv) (GQA paper, cited in
//    the TASP reference list).
//  * Partials restricted to a key range [kv_begin, kv_end) and their
//    log-sum-exp merge (the "partial attention computation" of the HSAP
//    abstract; Blockwise/Ring Attention, cited by TASP).
//  * Schedule properties: Ring AllGather visit order, zigzag chunking, and the
//    Hamiltonian decomposition of the complete directed graph into orthogonal
//    rings with the primitive decomposition of each chunk into P-1 pieces
//    (TASP abstract).
// Every floating-point step is in double precision; inputs may be given as
// float64, float32 or bfloat16 bit patterns and are widened exactly.
//
// Parity pins for every function live in the CPU test suite (brute force,
// closed forms, a library special case, merge and isolation invariants, and
// hand-written schedule fixtures). No function here is unpinned.

#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <cstdio>
#include <vector>
#include <algorithm>
#include <limits>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// Input dtype codes.
enum { DT_F64 = 0, DT_F32 = 1, DT_BF16 = 2 };

inline double widen(const void* base, int dtype, size_t idx) {
  if (dtype == DT_F64) return static_cast<const double*>(base)[idx];
  if (dtype == DT_F32) return static_cast<const float*>(base)[idx];
  // bfloat16: the upper 16 bits of an IEEE float32.
  uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return f;
}

// Index of the document that holds token t: the i with cu[i] <= t < cu[i+1].
int doc_of(const int32_t* cu, int ndocs, int t) {
  int lo = 0, hi = ndocs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

const double NEG_INF = -std::numeric_limits<double>::infinity();

}  // namespace

extern "C" {

// Validates a cu_seqlens array: cu[0] == 0, strictly increasing, cu[ndocs] == T.
// Returns 0 when valid.
int oracle_check_cu_seqlens(const int32_t* cu, int ndocs, int T) {
  if (ndocs < 1 || cu[0] != 0 || cu[ndocs] != T) return 1;
  for (int i = 0; i < ndocs; ++i)
    if (cu[i + 1] <= cu[i]) return 2;
  return 0;
}

int oracle_doc_of(const int32_t* cu, int ndocs, int t) { return doc_of(cu, ndocs, t); }

// Attention for the query tokens listed in `rows` (or every token when rows is
// NULL and nrows == T), over the keys in [kv_begin, kv_end) that are valid for
// that query. Layouts: q [T][Hq][d] (or [nrows][Hq][d] holding only the listed
// rows when q_rows_only is set), k and v [T][Hkv][d]. Outputs:
// o_out [nrows][Hq][d], lse_out [nrows][Hq]. A query with no valid key in the
// range gets LSE = -inf and O = 0. Returns 0 on success.
int oracle_attn(const void* q, const void* k, const void* v, int dtype,
                int T, int Hq, int Hkv, int d,
                const int32_t* cu, int ndocs, int causal, double scale,
                int kv_begin, int kv_end,
                const int32_t* rows, int nrows, int q_rows_only,
                double* o_out, double* lse_out, int nthreads) {
  if (T <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return 1;
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return 2;
  if (kv_begin < 0 || kv_end > T || kv_begin > kv_end) return 3;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int bad_row = 0;
#pragma omp parallel
  {
    std::vector<double> qi(d), s, acc(d);
#pragma omp for schedule(dynamic, 1)
    for (long long task = 0; task < static_cast<long long>(nrows) * Hq; ++task) {
      const int r = static_cast<int>(task / Hq);
      const int h = static_cast<int>(task % Hq);
      const int i = rows ? rows[r] : r;
      if (i < 0 || i >= T) { bad_row = 1; continue; }
      const int g = h / G;
      // V(i) restricted to [kv_begin, kv_end): the same document as i, and
      // j <= i when causal. Documents are contiguous token ranges, so the set
      // is one interval.
      const int D = doc_of(cu, ndocs, i);
      int j0 = std::max(cu[D], kv_begin);
      int j1 = std::min(cu[D + 1], kv_end);
      if (causal) j1 = std::min(j1, i + 1);
      double* o_row = o_out + (static_cast<size_t>(r) * Hq + h) * d;
      if (j1 <= j0) {
        for (int c = 0; c < d; ++c) o_row[c] = 0.0;
        lse_out[static_cast<size_t>(r) * Hq + h] = NEG_INF;
        continue;
      }
      const size_t qrow = q_rows_only ? static_cast<size_t>(r) : static_cast<size_t>(i);
      for (int c = 0; c < d; ++c) qi[c] = widen(q, dtype, (qrow * Hq + h) * d + c);
      s.resize(j1 - j0);
      double m = NEG_INF;
      for (int j = j0; j < j1; ++j) {
        const size_t kb = (static_cast<size_t>(j) * Hkv + g) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qi[c] * widen(k, dtype, kb + c);
        s[j - j0] = dot * scale;
        m = std::max(m, s[j - j0]);
      }
      double sum = 0.0;
      for (int j = j0; j < j1; ++j) sum += std::exp(s[j - j0] - m);
      const double lse = m + std::log(sum);
      std::fill(acc.begin(), acc.end(), 0.0);
      for (int j = j0; j < j1; ++j) {
        const double w = std::exp(s[j - j0] - lse);
        const size_t vb = (static_cast<size_t>(j) * Hkv + g) * d;
        for (int c = 0; c < d; ++c) acc[c] += w * widen(v, dtype, vb + c);
      }
      for (int c = 0; c < d; ++c) o_row[c] = acc[c];
      lse_out[static_cast<size_t>(r) * Hq + h] = lse;
    }
  }
  return bad_row ? 4 : 0;
}

// Log-sum-exp merge of two normalised partials over disjoint key sets:
//   L = M + log(exp(L1 - M) + exp(L2 - M)), M = max(L1, L2),
//   O = exp(L1 - L) O1 + exp(L2 - L) O2.
// A partial with L = -inf contributes nothing; two such stay -inf with O = 0.
// Layouts: o [n][d], lse [n] (n = rows x heads, any order shared by all four).
void oracle_lse_merge(const double* o1, const double* l1, const double* o2, const double* l2,
                      long long n, int d, double* o_out, double* l_out) {
  for (long long r = 0; r < n; ++r) {
    const double a = l1[r], b = l2[r];
    const double M = std::max(a, b);
    if (M == NEG_INF) {
      l_out[r] = NEG_INF;
      for (int c = 0; c < d; ++c) o_out[r * d + c] = 0.0;
      continue;
    }
    const double L = M + std::log(std::exp(a - M) + std::exp(b - M));
    const double wa = std::exp(a - L), wb = std::exp(b - L);
    for (int c = 0; c < d; ++c) o_out[r * d + c] = wa * o1[r * d + c] + wb * o2[r * d + c];
    l_out[r] = L;
  }
}

// Number of (query, key) pairs with query in [qa, qb) and key in [ka, kb)
// that the document and causal masks allow. Brute force over documents.
long long oracle_valid_pairs(const int32_t* cu, int ndocs, int causal,
                             int qa, int qb, int ka, int kb) {
  long long total = 0;
  for (int D = 0; D < ndocs; ++D) {
    const int r0 = std::max(qa, cu[D]), r1 = std::min(qb, cu[D + 1]);
    const int c0 = std::max(ka, cu[D]), c1 = std::min(kb, cu[D + 1]);
    if (r1 <= r0 || c1 <= c0) continue;
    if (!causal) { total += static_cast<long long>(r1 - r0) * (c1 - c0); continue; }
    for (int i = r0; i < r1; ++i) {
      const int hi = std::min(c1, i + 1);
      if (hi > c0) total += hi - c0;
    }
  }
  return total;
}

// ---------------------------------------------------------------------------
// Schedules.
//
// An item is 8 int32: rank, step, cycle, q_begin, q_end, kv_begin, kv_end,
// flags. The checks below re-derive what the schedule must contain without
// using the product's generator.

// Bounds of piece `idx` when [0, n) is cut into `parts` contiguous pieces and
// the first n mod parts pieces get one extra token.
static void split_bounds(int n, int parts, int idx, int* b, int* e) {
  const int base = n / parts, extra = n % parts;
  *b = idx * base + std::min(idx, extra);
  *e = *b + base + (idx < extra ? 1 : 0);
}

// Chunk boundaries out[0..P] of the chunking policies (load balancing,
// "HSAP: A Hierarchical Sequence-aware Parallelism for Hybrid-Context
// Generative Models", Methodology; whole-document sharding, FlashCP abstract
// on the same page), written from their definitions with per-token loops:
//   mode 0: the equal split above;
//   mode 1: with n(i) the keys row i attends and W(t) = n(0) + ... + n(t-1),
//           bound r = the smallest t with P * W(t) >= r * W(T);
//   mode 2: the mode-1 bounds, then for r = 1 .. P-1 in order: the document
//           start c (among cu[1 .. ndocs-1]) with |W(c) - W(bound r)| least
//           (the smaller c on a tie) replaces bound r if 16 P |W(c) - W(bound r)|
//           <= W(T) and c lies after the (already final) bound r-1; otherwise
//           bound r is raised to bound r-1 if it is below it.
// Returns 0, or nonzero for invalid arguments.
int oracle_chunk_bounds(int mode, int P, int T, const int32_t* cu, int ndocs, int causal, int32_t* out) {
  if (P < 1 || T < 0 || mode < 0 || mode > 2) return 1;
  if (T == 0) {
    for (int r = 0; r <= P; ++r) out[r] = 0;
    return 0;
  }
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return 2;
  if (mode == 0) {
    for (int r = 0; r < P; ++r) {
      int b, e;
      split_bounds(T, P, r, &b, &e);
      out[r] = b;
    }
    out[P] = T;
    return 0;
  }
  std::vector<long long> W(static_cast<size_t>(T) + 1, 0);
  for (int i = 0; i < T; ++i) {
    const int D = doc_of(cu, ndocs, i);
    const long long n = causal ? (i - cu[D] + 1) : (cu[D + 1] - cu[D]);
    W[i + 1] = W[i] + n;
  }
  out[0] = 0;
  for (int r = 1; r < P; ++r) {
    int t = 0;
    while (t < T && static_cast<long long>(P) * W[t] < static_cast<long long>(r) * W[T]) ++t;
    out[r] = t;
  }
  out[P] = T;
  if (mode == 2 && ndocs > 1) {
    for (int r = 1; r < P; ++r) {
      int best = -1;
      long long bdist = 0;
      for (int x = 1; x < ndocs; ++x) {
        const long long dist = std::llabs(W[cu[x]] - W[out[r]]);
        if (best < 0 || dist < bdist || (dist == bdist && cu[x] < best)) {
          best = cu[x];
          bdist = dist;
        }
      }
      if (16LL * P * bdist <= W[T] && best > out[r - 1]) out[r] = best;
      else if (out[r] < out[r - 1]) out[r] = out[r - 1];
    }
  }
  return 0;
}

// Writes the expected RING (kind 0) or ZIGZAG (kind 1) item list, before and
// after pruning of pairless items, in the canonical order: rank, then local Q
// piece in token order, then step. Returns the number of items, or -1 when
// the configuration is not allowed (zigzag needs T divisible by 2P).
// `out` may be NULL to count only. Flags are not produced (written 0).
long long oracle_closed_form_schedule(int kind, int P, int T, const int32_t* cu, int ndocs,
                                      int causal, int32_t* out, long long cap) {
  long long n = 0;
  auto emit = [&](int r, int s, int qa, int qb, int ka, int kb) {
    if (oracle_valid_pairs(cu, ndocs, causal, qa, qb, ka, kb) == 0) return;
    if (out && n < cap) {
      int32_t* it = out + n * 8;
      it[0] = r; it[1] = s; it[2] = 0; it[3] = qa; it[4] = qb; it[5] = ka; it[6] = kb; it[7] = 0;
    }
    ++n;
  };
  if (kind == 0) {
    for (int r = 0; r < P; ++r) {
      int qa, qb;
      split_bounds(T, P, r, &qa, &qb);
      for (int s = 0; s < P; ++s) {
        const int src = ((r - s) % P + P) % P;
        int ka, kb;
        split_bounds(T, P, src, &ka, &kb);
        emit(r, s, qa, qb, ka, kb);
      }
    }
    return n;
  }
  if (kind == 1) {
    if (T % (2 * P) != 0) return -1;
    const int c = T / (2 * P);
    for (int r = 0; r < P; ++r) {
      const int mine[2] = {r, 2 * P - 1 - r};  // r < 2P-1-r, so token order
      for (int a = 0; a < 2; ++a) {
        for (int s = 0; s < P; ++s) {
          const int src = ((r - s) % P + P) % P;
          const int theirs[2] = {src, 2 * P - 1 - src};
          for (int b = 0; b < 2; ++b)
            emit(r, s, mine[a] * c, (mine[a] + 1) * c, theirs[b] * c, (theirs[b] + 1) * c);
        }
      }
    }
    return n;
  }
  return -1;
}

// Checks that succ (P-1 rows of P successors) is a decomposition of the
// complete directed graph on P vertices into P-1 arc-disjoint directed
// Hamiltonian cycles. Returns 0 when it is; otherwise a nonzero code:
// 1 bad vertex id or self loop, 2 a row is not one P-cycle, 3 an arc repeats.
int oracle_check_hamiltonian(int P, const int32_t* succ) {
  if (P < 2) return 0;
  std::vector<int> used(static_cast<size_t>(P) * P, 0);
  for (int c = 0; c < P - 1; ++c) {
    const int32_t* sc = succ + static_cast<size_t>(c) * P;
    for (int u = 0; u < P; ++u)
      if (sc[u] < 0 || sc[u] >= P || sc[u] == u) return 1;
    // Walk from 0: a Hamiltonian cycle returns to 0 after exactly P arcs and
    // visits every vertex once.
    std::vector<int> seen(P, 0);
    int u = 0;
    for (int step = 0; step < P; ++step) {
      if (seen[u]) return 2;
      seen[u] = 1;
      u = sc[u];
    }
    if (u != 0) return 2;
    for (int w = 0; w < P; ++w) {
      int& cnt = used[static_cast<size_t>(w) * P + sc[w]];
      if (++cnt > 1) return 3;
    }
  }
  // P-1 cycles of P arcs, none repeated, no self loops: all P(P-1) arcs used.
  return 0;
}

// Checks an item list against the method's requirements. Returns 0 when all
// hold, else a code, and writes a one-line reason into msg.
//   * every item lies inside [0, T), has begin < end and at least one valid
//     (query, key) pair (the sequence-aware pruning: no item without work);
//   * the Q ranges: rank r of RING/TASP owns chunk r of P; rank r of ZIGZAG
//     owns chunks r and 2P-1-r of 2P;
//   * for each rank and each of its Q ranges, the item key ranges are pairwise
//     disjoint, and together they contain every key that some query of the
//     range may attend (so each valid pair is computed exactly once);
//   * TASP (kind 2): step 0 is the local chunk; at step t >= 1 the item of
//     cycle c holds piece c of chunk pred_c^t(r), where pred_c inverts row c
//     of succ and piece c is cut by the "first n mod (P-1) pieces get one
//     more token" rule; succ must pass oracle_check_hamiltonian.
// If brute is nonzero, the exact-once property is additionally checked by
// counting every valid pair (use only for small T).
int oracle_check_schedule(int kind, int P, int T, const int32_t* cu, int ndocs, int causal,
                          const int32_t* items, long long n_items, const int32_t* succ,
                          int brute, char* msg, int msg_len, const int32_t* bounds) {
  auto fail = [&](int code, const char* fmt, long long a, long long b) {
    if (msg && msg_len > 0) std::snprintf(msg, msg_len, fmt, a, b);
    return code;
  };
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return fail(1, "bad cu_seqlens %lld %lld", 0, 0);
  if (P < 1) return fail(1, "bad P %lld %lld", P, 0);
  if (bounds && (kind == 1 || bounds[0] != 0 || bounds[P] != T)) return fail(1, "bad bounds %lld %lld", kind, P);
  if (bounds)
    for (int r = 0; r < P; ++r)
      if (bounds[r + 1] < bounds[r]) return fail(1, "bounds decrease at %lld %lld", r, bounds[r]);
  // Chunk x of the RING / TASP split: the given bounds, else the equal split.
  auto chunk_of = [&](int x, int* b, int* e) {
    if (bounds) {
      *b = bounds[x];
      *e = bounds[x + 1];
    } else {
      split_bounds(T, P, x, b, e);
    }
  };
  // Owned Q ranges per rank.
  std::vector<std::vector<std::pair<int, int>>> own(P);
  for (int r = 0; r < P; ++r) {
    if (kind == 1) {
      if (T % (2 * P) != 0) return fail(1, "zigzag needs T %% 2P == 0 (T=%lld, P=%lld)", T, P);
      const int c = T / (2 * P);
      own[r].push_back({r * c, (r + 1) * c});
      own[r].push_back({(2 * P - 1 - r) * c, (2 * P - r) * c});
    } else {
      int a, b;
      chunk_of(r, &a, &b);
      if (a < b) own[r].push_back({a, b});
    }
  }
  if (kind == 2 && P >= 2) {
    const int hc = oracle_check_hamiltonian(P, succ);
    if (hc != 0) return fail(2, "not a Hamiltonian decomposition (code %lld) %lld", hc, 0);
  }
  // pred tables for TASP.
  std::vector<int> pred;
  if (kind == 2 && P >= 2) {
    pred.assign(static_cast<size_t>(P - 1) * P, -1);
    for (int c = 0; c < P - 1; ++c)
      for (int u = 0; u < P; ++u) pred[static_cast<size_t>(c) * P + succ[static_cast<size_t>(c) * P + u]] = u;
  }
  // Per (rank, q range): list of key ranges.
  std::vector<std::vector<std::vector<std::pair<int, int>>>> keys(P);
  for (int r = 0; r < P; ++r) keys[r].resize(own[r].size());
  for (long long x = 0; x < n_items; ++x) {
    const int32_t* it = items + x * 8;
    const int r = it[0], s = it[1], c = it[2], qa = it[3], qb = it[4], ka = it[5], kb = it[6];
    if (r < 0 || r >= P) return fail(3, "item %lld: bad rank %lld", x, r);
    if (!(0 <= qa && qa < qb && qb <= T && 0 <= ka && ka < kb && kb <= T))
      return fail(3, "item %lld: bad ranges (q_begin %lld)", x, qa);
    if (oracle_valid_pairs(cu, ndocs, causal, qa, qb, ka, kb) == 0)
      return fail(4, "item %lld has no valid pair (rank %lld)", x, r);
    int which = -1;
    for (size_t w = 0; w < own[r].size(); ++w)
      if (own[r][w].first == qa && own[r][w].second == qb) which = static_cast<int>(w);
    if (which < 0) return fail(5, "item %lld: Q range not owned by rank %lld", x, r);
    keys[r][which].push_back({ka, kb});
    if (kind == 2) {
      int ea, eb;
      if (s == 0) {
        chunk_of(r, &ea, &eb);
      } else {
        if (P < 2 || c < 0 || c >= P - 1 || s >= P) return fail(6, "item %lld: bad step/cycle %lld", x, s);
        int src = r;
        for (int t = 0; t < s; ++t) src = pred[static_cast<size_t>(c) * P + src];
        int cb, ce;
        chunk_of(src, &cb, &ce);
        int pb, pe;
        split_bounds(ce - cb, P - 1, c, &pb, &pe);
        ea = cb + pb;
        eb = cb + pe;
      }
      if (ka != ea || kb != eb) return fail(7, "item %lld: TASP key range starts %lld, expected", x, ka);
    }
  }
  // Coverage: disjoint and complete for each owned Q range.
  for (int r = 0; r < P; ++r) {
    for (size_t w = 0; w < own[r].size(); ++w) {
      auto ks = keys[r][w];
      std::sort(ks.begin(), ks.end());
      for (size_t y = 1; y < ks.size(); ++y)
        if (ks[y].first < ks[y - 1].second) return fail(8, "rank %lld: overlapping key ranges at %lld", r, ks[y].first);
      const int qa = own[r][w].first, qb = own[r][w].second;
      // Keys some query of [qa, qb) may attend: per document D meeting the
      // range, [cu[D], cu[D+1]) (non-causal) or [cu[D], min(cu[D+1], qb)).
      for (int D = 0; D < ndocs; ++D) {
        if (cu[D + 1] <= qa || cu[D] >= qb) continue;
        const int need0 = cu[D];
        const int need1 = causal ? std::min(cu[D + 1], qb) : cu[D + 1];
        // Walk the sorted disjoint ranges and make sure [need0, need1) is covered.
        int pos = need0;
        for (const auto& kr : ks) {
          if (kr.second <= pos) continue;
          if (kr.first > pos) break;
          pos = kr.second;
          if (pos >= need1) break;
        }
        if (pos < need1) return fail(9, "rank %lld: key %lld needed but not covered", r, pos);
      }
    }
  }
  if (brute) {
    std::vector<int> doc(T);
    for (int t = 0; t < T; ++t) doc[t] = doc_of(cu, ndocs, t);
    std::vector<uint8_t> cnt(static_cast<size_t>(T) * T, 0);
    for (long long x = 0; x < n_items; ++x) {
      const int32_t* it = items + x * 8;
      for (int i = it[3]; i < it[4]; ++i)
        for (int j = it[5]; j < it[6]; ++j) {
          if (doc[i] != doc[j] || (causal && j > i)) continue;
          uint8_t& cc = cnt[static_cast<size_t>(i) * T + j];
          if (cc < 255) ++cc;
        }
    }
    for (int i = 0; i < T; ++i)
      for (int j = 0; j < T; ++j) {
        const bool valid = (doc[i] == doc[j]) && (!causal || j <= i);
        const uint8_t cc = cnt[static_cast<size_t>(i) * T + j];
        if (valid && cc != 1) return fail(10, "pair (%lld, %lld) not computed exactly once", i, j);
      }
  }
  return 0;
}

int oracle_link_bytes(int kind, int P, int T, const int32_t* cu, int ndocs, int causal,
                      const int32_t* succ, long long bytes_per_token, int needed_only,
                      long long* out);

// Communication of a two-level schedule, restated token by token and head by
// head: token t belongs to group g (its chunk of the R-way split, or the pair
// of the 2R-way split for zigzag) and, by its position in the group's tokens
// cut into U parts, to rank g*U + u. For every query head h of a slice u'
// != u the token's q (before) and o (after) cross the links u -> u' and
// u' -> u; for every key/value head a slice u' != u uses, its k and v cross
// u -> u'. The Inter-SP part is oracle_link_bytes of the R groups, with the
// key/value heads each slice uses, placed on the links between the ranks of
// that slice. Output layout as the library's sp_schedule_link_bytes_hier.
int oracle_link_bytes_hier(int kind, int R, int U, int T, const int32_t* cu, int ndocs, int causal,
                           const int32_t* succ, int Hq, int Hkv, int d, int eb, int needed_only,
                           long long* intra, long long* inter) {
  if (R < 1 || U < 1 || Hq % U != 0 || Hq % Hkv != 0) return 1;
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return 2;
  const int P = R * U, hs = Hq / U, G = Hq / Hkv;
  const size_t PP = static_cast<size_t>(P) * P;
  for (size_t i = 0; i < PP; ++i) intra[i] = 0;
  // Tokens of each group, in token order.
  std::vector<std::vector<int>> toks(R);
  for (int t = 0; t < T; ++t) {
    int g;
    if (kind == 1) {
      const int c = t / (T / (2 * R));
      g = c < R ? c : 2 * R - 1 - c;
    } else {
      g = 0;
      for (int x = 0; x < R; ++x) {
        int b, e;
        split_bounds(T, R, x, &b, &e);
        if (t >= b && t < e) g = x;
      }
    }
    toks[g].push_back(t);
  }
  // Key/value heads used by each slice.
  std::vector<std::vector<int>> uses(U, std::vector<int>(Hkv, 0));
  for (int h = 0; h < Hq; ++h) uses[h / hs][h / G] = 1;
  for (int g = 0; g < R; ++g) {
    const int n_g = static_cast<int>(toks[g].size());
    for (int p = 0; p < n_g; ++p) {
      int u = 0;
      for (int x = 0; x < U; ++x) {
        int b, e;
        split_bounds(n_g, U, x, &b, &e);
        if (p >= b && p < e) u = x;
      }
      const int owner = g * U + u;
      for (int h = 0; h < Hq; ++h) {
        const int v = h / hs;
        if (v == u) continue;
        intra[static_cast<size_t>(owner) * P + (g * U + v)] += static_cast<long long>(d) * eb;  // q
        intra[static_cast<size_t>(g * U + v) * P + owner] += static_cast<long long>(d) * eb;    // o
      }
      for (int v = 0; v < U; ++v) {
        if (v == u) continue;
        for (int kvh = 0; kvh < Hkv; ++kvh)
          if (uses[v][kvh]) intra[static_cast<size_t>(owner) * P + (g * U + v)] += 2LL * d * eb;  // k, v
      }
    }
  }
  if (R == 1) return 0;
  for (size_t i = 0; i < static_cast<size_t>(R - 1) * PP; ++i) inter[i] = 0;
  std::vector<long long> grp(static_cast<size_t>(R - 1) * R * R);
  for (int v = 0; v < U; ++v) {
    long long nkv = 0;
    for (int kvh = 0; kvh < Hkv; ++kvh) nkv += uses[v][kvh];
    const int rc = oracle_link_bytes(kind, R, T, cu, ndocs, causal, succ, 2 * nkv * d * eb, needed_only,
                                     grp.data());
    if (rc != 0) return 10 + rc;
    for (int t = 0; t < R - 1; ++t)
      for (int a = 0; a < R; ++a)
        for (int b = 0; b < R; ++b)
          inter[static_cast<size_t>(t) * PP + static_cast<size_t>(a * U + v) * P + (b * U + v)] =
              grp[static_cast<size_t>(t) * R * R + static_cast<size_t>(a) * R + b];
  }
  return 0;
}

// Checks a two-level schedule on P = R * U ranks (Inter-SP schedule of kind
// `kind` over R groups; inside group g, rank g*U + u takes query heads
// [u Hq/U, (u+1) Hq/U)): every item's head range must be its rank's slice,
// and for each u the items of ranks g*U + u, renumbered g, must form a valid
// R-rank schedule by oracle_check_schedule (same succ, bounds and brute
// options). Then every (query, key, head) triple the mask allows is covered
// exactly once: each head lies in exactly one slice, and within a slice the
// R-rank schedule covers every valid pair once. Returns 0 or a nonzero code
// (20 bad arguments, 21 bad rank, 22 wrong head range, 30 + the code of the
// failing slice's check).
int oracle_check_hier_schedule(int kind, int R, int U, int Hq, int T, const int32_t* cu, int ndocs,
                               int causal, const int32_t* items, const int32_t* heads, long long n_items,
                               const int32_t* succ, int brute, char* msg, int msg_len,
                               const int32_t* bounds) {
  auto fail = [&](int code, const char* fmt, long long a, long long b) {
    if (msg && msg_len > 0) std::snprintf(msg, msg_len, fmt, a, b);
    return code;
  };
  if (R < 1 || U < 1 || Hq < 1 || Hq % U != 0) return fail(20, "bad R/U/Hq %lld %lld", R, U);
  const int hs = Hq / U;
  std::vector<std::vector<int32_t>> slice(U);
  for (long long x = 0; x < n_items; ++x) {
    const int32_t* it = items + x * 8;
    const int r = it[0];
    if (r < 0 || r >= R * U) return fail(21, "item %lld: bad rank %lld", x, r);
    const int u = r % U;
    if (heads[2 * x] != u * hs || heads[2 * x + 1] != (u + 1) * hs)
      return fail(22, "item %lld: head range starts at %lld", x, heads[2 * x]);
    for (int c = 0; c < 8; ++c) slice[u].push_back(c == 0 ? r / U : it[c]);
  }
  for (int u = 0; u < U; ++u) {
    const long long m = static_cast<long long>(slice[u].size() / 8);
    char sub[200];
    const int rc = oracle_check_schedule(kind, R, T, cu, ndocs, causal, slice[u].data(), m, succ, brute, sub,
                                         sizeof sub, bounds);
    if (rc != 0) {
      if (msg && msg_len > 0) std::snprintf(msg, msg_len, "head slice %d: %s", u, sub);
      return 30 + rc;
    }
  }
  return 0;
}

// Gradients of the masked attention (the backward of the operation above):
// with P_ij = exp(s_ij - LSE_i) over the valid keys j of query i,
//   dV_j  = sum_i P_ij dO_i,              dP_ij = dO_i . v_j,
//   D_i   = sum_j P_ij dP_ij (= dO_i . O_i),  dS_ij = P_ij (dP_ij - D_i),
//   dQ_i  = scale sum_j dS_ij k_j,        dK_j  = scale sum_i dS_ij q_i,
// where dK and dV of key/value head g sum over the query heads h with
// h / (Hq/Hkv) == g. LSE and O are recomputed here in fp64 from q, k, v.
// Layouts as oracle_attn; dq_out [T][Hq][d], dk_out / dv_out [T][Hkv][d].
int oracle_attn_backward(const void* q, const void* k, const void* v, const void* dout, int dtype,
                         int T, int Hq, int Hkv, int d, const int32_t* cu, int ndocs, int causal,
                         double scale, double* dq_out, double* dk_out, double* dv_out,
                         int nthreads) {
  if (T <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return 1;
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return 2;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  for (size_t x = 0; x < static_cast<size_t>(T) * Hq * d; ++x) dq_out[x] = 0.0;
  for (size_t x = 0; x < static_cast<size_t>(T) * Hkv * d; ++x) dk_out[x] = dv_out[x] = 0.0;
  // One key/value head per task, so dK and dV of that head have one writer.
#pragma omp parallel for schedule(dynamic, 1)
  for (int g = 0; g < Hkv; ++g) {
    std::vector<double> qi(d), doi(d), s, p, o(d);
    for (int h = g * G; h < (g + 1) * G; ++h) {
      for (int i = 0; i < T; ++i) {
        const int D = doc_of(cu, ndocs, i);
        const int j0 = cu[D];
        const int j1 = causal ? std::min(cu[D + 1], i + 1) : cu[D + 1];
        const size_t qb = (static_cast<size_t>(i) * Hq + h) * d;
        for (int c = 0; c < d; ++c) {
          qi[c] = widen(q, dtype, qb + c);
          doi[c] = widen(dout, dtype, qb + c);
        }
        s.resize(j1 - j0);
        p.resize(j1 - j0);
        double m = NEG_INF;
        for (int j = j0; j < j1; ++j) {
          const size_t kb = (static_cast<size_t>(j) * Hkv + g) * d;
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += qi[c] * widen(k, dtype, kb + c);
          s[j - j0] = dot * scale;
          m = std::max(m, s[j - j0]);
        }
        double sum = 0.0;
        for (int j = j0; j < j1; ++j) sum += std::exp(s[j - j0] - m);
        const double lse = m + std::log(sum);
        std::fill(o.begin(), o.end(), 0.0);
        for (int j = j0; j < j1; ++j) {
          p[j - j0] = std::exp(s[j - j0] - lse);
          const size_t vb = (static_cast<size_t>(j) * Hkv + g) * d;
          for (int c = 0; c < d; ++c) o[c] += p[j - j0] * widen(v, dtype, vb + c);
        }
        double Di = 0.0;
        for (int c = 0; c < d; ++c) Di += doi[c] * o[c];
        for (int j = j0; j < j1; ++j) {
          const size_t kb = (static_cast<size_t>(j) * Hkv + g) * d;
          double dp = 0.0;
          for (int c = 0; c < d; ++c) dp += doi[c] * widen(v, dtype, kb + c);
          const double pij = p[j - j0];
          const double ds = pij * (dp - Di);
          for (int c = 0; c < d; ++c) {
            dv_out[kb + c] += pij * doi[c];
            dq_out[qb + c] += scale * ds * widen(k, dtype, kb + c);
            dk_out[kb + c] += scale * ds * qi[c];
          }
        }
      }
    }
  }
  return 0;
}

// The same gradients restricted to chosen outputs, for checking a large
// problem on samples: dQ of the listed query rows, and dK, dV of the listed
// keys. Each value follows the definitions above term by term; a query's LSE
// and D are recomputed from q, k, v over its own valid keys (once per query
// and head, since several keys share the queries that attend them).
//  qrows[nq] -> dq_rows [nq][Hq][d];  krows[nk] -> dk_rows, dv_rows [nk][Hkv][d].
namespace {

struct RowStats {
  double lse, D;
};

// LSE and D = dO . O of query i under head h (g = its key/value head).
RowStats row_stats(const void* q, const void* k, const void* v, const void* dout, int dtype, int Hq,
                   int Hkv, int d, const int32_t* cu, int ndocs, int causal, double scale, int i,
                   int h, int g) {
  const int D = doc_of(cu, ndocs, i);
  const int j0 = cu[D];
  const int j1 = causal ? std::min(cu[D + 1], i + 1) : cu[D + 1];
  const size_t qb = (static_cast<size_t>(i) * Hq + h) * d;
  std::vector<double> s(j1 - j0), o(d, 0.0);
  double m = NEG_INF;
  for (int j = j0; j < j1; ++j) {
    const size_t kb = (static_cast<size_t>(j) * Hkv + g) * d;
    double dot = 0.0;
    for (int c = 0; c < d; ++c) dot += widen(q, dtype, qb + c) * widen(k, dtype, kb + c);
    s[j - j0] = dot * scale;
    m = std::max(m, s[j - j0]);
  }
  double sum = 0.0;
  for (int j = j0; j < j1; ++j) sum += std::exp(s[j - j0] - m);
  RowStats r;
  r.lse = m + std::log(sum);
  for (int j = j0; j < j1; ++j) {
    const double pij = std::exp(s[j - j0] - r.lse);
    const size_t vb = (static_cast<size_t>(j) * Hkv + g) * d;
    for (int c = 0; c < d; ++c) o[c] += pij * widen(v, dtype, vb + c);
  }
  r.D = 0.0;
  for (int c = 0; c < d; ++c) r.D += widen(dout, dtype, qb + c) * o[c];
  return r;
}

// P_ij, dP_ij for query i (head h) and key j (key/value head g).
void pair_terms(const void* q, const void* k, const void* v, const void* dout, int dtype, int Hq,
                int Hkv, int d, double scale, int i, int h, int j, int g, const RowStats& st,
                double* p, double* dp) {
  const size_t qb = (static_cast<size_t>(i) * Hq + h) * d;
  const size_t kb = (static_cast<size_t>(j) * Hkv + g) * d;
  double dot = 0.0, dpd = 0.0;
  for (int c = 0; c < d; ++c) {
    dot += widen(q, dtype, qb + c) * widen(k, dtype, kb + c);
    dpd += widen(dout, dtype, qb + c) * widen(v, dtype, kb + c);
  }
  *p = std::exp(dot * scale - st.lse);
  *dp = dpd;
}

}  // namespace

int oracle_attn_backward_sampled(const void* q, const void* k, const void* v, const void* dout,
                                 int dtype, int T, int Hq, int Hkv, int d, const int32_t* cu,
                                 int ndocs, int causal, double scale, const int32_t* qrows, int nq,
                                 double* dq_rows, const int32_t* krows, int nk, double* dk_rows,
                                 double* dv_rows, int nthreads) {
  if (T <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || nq < 0 || nk < 0) return 1;
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return 2;
  for (int x = 0; x < nq; ++x)
    if (qrows[x] < 0 || qrows[x] >= T) return 3;
  for (int x = 0; x < nk; ++x)
    if (krows[x] < 0 || krows[x] >= T) return 3;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  // dQ_i = scale sum_j dS_ij k_j over the valid keys of row i.
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int x = 0; x < nq; ++x)
    for (int h = 0; h < Hq; ++h) {
      const int i = qrows[x], g = h / G;
      const RowStats st = row_stats(q, k, v, dout, dtype, Hq, Hkv, d, cu, ndocs, causal, scale, i, h, g);
      const int D = doc_of(cu, ndocs, i);
      const int j1 = causal ? std::min(cu[D + 1], i + 1) : cu[D + 1];
      double* out = dq_rows + (static_cast<size_t>(x) * Hq + h) * d;
      for (int c = 0; c < d; ++c) out[c] = 0.0;
      for (int j = cu[D]; j < j1; ++j) {
        double p, dp;
        pair_terms(q, k, v, dout, dtype, Hq, Hkv, d, scale, i, h, j, g, st, &p, &dp);
        const double ds = p * (dp - st.D);
        const size_t kb = (static_cast<size_t>(j) * Hkv + g) * d;
        for (int c = 0; c < d; ++c) out[c] += scale * ds * widen(k, dtype, kb + c);
      }
    }
  if (nk == 0) return 0;
  // The queries that attend some listed key, and their statistics per head.
  std::vector<int> need;
  {
    std::vector<char> mark(T, 0);
    for (int x = 0; x < nk; ++x) {
      const int j = krows[x];
      const int D = doc_of(cu, ndocs, j);
      for (int i = causal ? j : cu[D]; i < cu[D + 1]; ++i) mark[i] = 1;
    }
    for (int i = 0; i < T; ++i)
      if (mark[i]) need.push_back(i);
  }
  std::vector<int> slot(T, -1);
  for (size_t n = 0; n < need.size(); ++n) slot[need[n]] = static_cast<int>(n);
  std::vector<RowStats> stats(need.size() * Hq);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (long long n = 0; n < static_cast<long long>(need.size()); ++n)
    for (int h = 0; h < Hq; ++h)
      stats[n * Hq + h] = row_stats(q, k, v, dout, dtype, Hq, Hkv, d, cu, ndocs, causal, scale,
                                    need[n], h, h / G);
  // dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij q_i over the queries
  // attending j and the query heads of j's key/value head.
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int x = 0; x < nk; ++x)
    for (int g = 0; g < Hkv; ++g) {
      const int j = krows[x];
      const int D = doc_of(cu, ndocs, j);
      double* dk = dk_rows + (static_cast<size_t>(x) * Hkv + g) * d;
      double* dv = dv_rows + (static_cast<size_t>(x) * Hkv + g) * d;
      for (int c = 0; c < d; ++c) dk[c] = dv[c] = 0.0;
      for (int h = g * G; h < (g + 1) * G; ++h)
        for (int i = causal ? j : cu[D]; i < cu[D + 1]; ++i) {
          const RowStats& st = stats[static_cast<size_t>(slot[i]) * Hq + h];
          double p, dp;
          pair_terms(q, k, v, dout, dtype, Hq, Hkv, d, scale, i, h, j, g, st, &p, &dp);
          const double ds = p * (dp - st.D);
          const size_t qb = (static_cast<size_t>(i) * Hq + h) * d;
          for (int c = 0; c < d; ++c) {
            dv[c] += p * widen(dout, dtype, qb + c);
            dk[c] += scale * ds * widen(q, dtype, qb + c);
          }
        }
    }
  return 0;
}

// Communication model of a schedule, stated from the receiving side: in
// iteration t (1..P-1) of the AllGather, what does each rank receive and from
// whom (TASP abstract: Ring AllGather = P-1 iterations of ring transfers; TASP
// = the same AllGather split into one piece per Hamiltonian ring per
// iteration). out[(t-1)*P*P + src*P + dst] += bytes. With needed_only, a
// reception counts only if the receiver or a rank after it on the same ring
// (within the iterations that remain) has a valid pair with the block.
int oracle_link_bytes(int kind, int P, int T, const int32_t* cu, int ndocs, int causal,
                      const int32_t* succ, long long bytes_per_token, int needed_only,
                      long long* out) {
  if (P < 2) return 0;
  if (oracle_check_cu_seqlens(cu, ndocs, T) != 0) return 1;
  if (kind == 1 && T % (2 * P) != 0) return 2;
  const size_t PP = static_cast<size_t>(P) * P;
  for (size_t i = 0; i < static_cast<size_t>(P - 1) * PP; ++i) out[i] = 0;
  auto chunk = [&](int x, int* a, int* b) { split_bounds(T, P, x, a, b); };
  // Q ranges of rank r.
  auto qranges = [&](int r, std::vector<std::pair<int, int>>& q) {
    q.clear();
    if (kind == 1) {
      const int c = T / (2 * P);
      q.push_back({r * c, (r + 1) * c});
      q.push_back({(2 * P - 1 - r) * c, (2 * P - r) * c});
    } else {
      int a, b;
      chunk(r, &a, &b);
      q.push_back({a, b});
    }
  };
  auto wants = [&](int r, int ka, int kb) {
    std::vector<std::pair<int, int>> q;
    qranges(r, q);
    for (auto& x : q)
      if (oracle_valid_pairs(cu, ndocs, causal, x.first, x.second, ka, kb) > 0) return true;
    return false;
  };
  for (int t = 1; t < P; ++t) {
    for (int r = 0; r < P; ++r) {
      if (kind == 0 || kind == 1) {
        const int src_rank = ((r - t) % P + P) % P;  // whose chunk(s) arrive
        const int from = (r + P - 1) % P;
        std::vector<std::pair<int, int>> blocks;
        if (kind == 0) {
          int a, b;
          chunk(src_rank, &a, &b);
          blocks.push_back({a, b});
        } else {
          qranges(src_rank, blocks);
        }
        for (auto& bl : blocks) {
          bool keep = !needed_only;
          for (int k = 0; !keep && t + k <= P - 1; ++k)
            if (wants((r + k) % P, bl.first, bl.second)) keep = true;
          if (keep)
            out[static_cast<size_t>(t - 1) * PP + static_cast<size_t>(from) * P + r] +=
                (bl.second - bl.first) * bytes_per_token;
        }
      } else {
        for (int c = 0; c < P - 1; ++c) {
          const int32_t* sc = succ + static_cast<size_t>(c) * P;
          // predecessor of r on ring c, and the rank t hops upstream
          int from = -1;
          for (int u = 0; u < P; ++u)
            if (sc[u] == r) from = u;
          int src_rank = r;
          for (int h = 0; h < t; ++h)
            for (int u = 0; u < P; ++u)
              if (sc[u] == src_rank) { src_rank = u; break; }
          int cb, ce, pb, pe;
          chunk(src_rank, &cb, &ce);
          split_bounds(ce - cb, P - 1, c, &pb, &pe);
          const int ka = cb + pb, kb = cb + pe;
          if (kb <= ka) continue;
          bool keep = !needed_only;
          int v = r;
          for (int k = 0; !keep && t + k <= P - 1; ++k) {
            if (wants(v, ka, kb)) keep = true;
            v = sc[v];
          }
          if (keep)
            out[static_cast<size_t>(t - 1) * PP + static_cast<size_t>(from) * P + r] +=
                (kb - ka) * bytes_per_token;
        }
      }
    }
  }
  return 0;
}

}  // extern "C"
