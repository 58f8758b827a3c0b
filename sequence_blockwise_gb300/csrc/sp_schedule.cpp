// Host-side chunk-visit schedules for virtual sequence-parallel ranks.
//
// RING follows the Ring AllGather order of Ring Attention, ZIGZAG its
// Zigzag-Ring variant, and TASP the topology decomposition (P-1 arc-disjoint
// directed Hamiltonian cycles of the complete digraph on P ranks) with the
// primitive decomposition (each KV chunk cut into P-1 pieces, piece c relayed
// on ring c) — "TASP: Topology-aware Sequence Parallelism", abstract. Items
// without a valid (query, key) pair are pruned, the plainest reading of
// sequence-aware scheduling of incomplete QKV on packed sequences ("HSAP",
// abstract and method summary).
//
// The Hamiltonian decomposition is found by a seeded randomized search: whole
// cycles are drawn by depth-first search with a fewest-exits-first order, and
// the last two cycles are split exactly from the 2-regular remainder by
// enumerating its perfect matchings. Everything is integer arithmetic, so the
// result is identical on every host for a given (P, seed). Complete digraphs
// on 4 and 6 vertices have no such decomposition (a result of graph theory,
// not of the pages); every other P does.

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/sp_attn.h"

namespace {

struct Rng {  // splitmix64
  uint64_t s;
  explicit Rng(uint64_t seed) : s(seed) {}
  uint64_t next() {
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  uint32_t below(uint32_t n) { return static_cast<uint32_t>(next() % n); }
};

inline int popc(uint64_t x) { return __builtin_popcountll(x); }
inline uint64_t bit(int v) { return 1ull << v; }

// Randomised DFS for a directed Hamiltonian cycle through vertex 0 in the
// digraph given by out/in masks. Returns true and fills succ on success.
struct HamSearch {
  int P;
  const uint64_t* out;
  const uint64_t* in;
  Rng* rng;
  long long budget;
  std::vector<int> path;

  bool feasible(uint64_t unvisited, int cur) const {
    // Every unvisited vertex still needs an entry from cur/unvisited and an
    // exit to unvisited/vertex 0.
    uint64_t from = unvisited | bit(cur);
    uint64_t to = unvisited | bit(0);
    for (uint64_t m = unvisited; m; m &= m - 1) {
      int w = __builtin_ctzll(m);
      if (!(in[w] & from) || !(out[w] & to)) return false;
    }
    return true;
  }

  bool dfs(int cur, uint64_t unvisited) {
    if (--budget < 0) return false;
    if (!unvisited) return (out[cur] & bit(0)) != 0;
    uint64_t cand = out[cur] & unvisited;
    if (!cand) return false;
    int vs[64], keys[64], n = 0;
    for (uint64_t m = cand; m; m &= m - 1) {
      int v = __builtin_ctzll(m);
      vs[n] = v;
      // fewest onward exits first, random tie break
      keys[n] = popc(out[v] & (unvisited & ~bit(v))) * 1024 + static_cast<int>(rng->below(1024));
      ++n;
    }
    for (int a = 1; a < n; ++a)
      for (int b = a; b > 0 && keys[b] < keys[b - 1]; --b) {
        std::swap(keys[b], keys[b - 1]);
        std::swap(vs[b], vs[b - 1]);
      }
    for (int x = 0; x < n; ++x) {
      int v = vs[x];
      uint64_t rest = unvisited & ~bit(v);
      if (rest && !feasible(rest, v)) continue;
      path.push_back(v);
      if (dfs(v, rest)) return true;
      path.pop_back();
      if (budget < 0) return false;
    }
    return false;
  }

  bool run(std::vector<int>& succ) {
    path.clear();
    path.push_back(0);
    uint64_t all = (P == 64) ? ~0ull : (bit(P) - 1);
    if (!dfs(0, all & ~bit(0))) return false;
    succ.assign(P, -1);
    for (int i = 0; i < P; ++i) succ[path[i]] = path[(i + 1) % P];
    return true;
  }
};

bool single_cycle(const std::vector<int>& succ) {
  const int P = static_cast<int>(succ.size());
  int u = 0;
  for (int i = 1; i < P; ++i) {
    u = succ[u];
    if (u == 0) return false;
  }
  return succ[u] == 0;
}

// Splits a 2-in/2-out regular digraph into two Hamiltonian cycles, if possible.
bool split_two(int P, const uint64_t* out, std::vector<int>& a, std::vector<int>& b) {
  // Components of the bipartite (tail, head) graph: alternate "first arc of a
  // tail" / "other in-arc of its head" until the walk closes.
  std::vector<std::vector<std::pair<int, int>>> comps;  // arcs in walk order
  std::vector<char> seen_tail(P, 0);
  std::vector<int> in_a(P, -1), in_b(P, -1);  // the two tails entering each head
  for (int u = 0; u < P; ++u)
    for (uint64_t m = out[u]; m; m &= m - 1) {
      int v = __builtin_ctzll(m);
      if (in_a[v] < 0) in_a[v] = u; else in_b[v] = u;
    }
  for (int u0 = 0; u0 < P; ++u0) {
    if (seen_tail[u0]) continue;
    std::vector<std::pair<int, int>> arcs;
    int u = u0;
    int v = __builtin_ctzll(out[u]);
    while (true) {
      seen_tail[u] = 1;
      arcs.push_back({u, v});               // even position: option 0
      int u2 = (in_a[v] == u) ? in_b[v] : in_a[v];
      uint64_t o2 = out[u2] & ~bit(v);
      int v2 = __builtin_ctzll(o2);
      arcs.push_back({u2, v});              // odd position: option 1
      seen_tail[u2] = 1;
      if (u2 == u0) break;
      u = u2;
      v = v2;
    }
    comps.push_back(arcs);
  }
  const int nc = static_cast<int>(comps.size());
  if (nc > 22) return false;
  a.assign(P, -1);
  b.assign(P, -1);
  for (uint32_t mask = 0; mask < (1u << nc); ++mask) {
    for (int c = 0; c < nc; ++c) {
      const int pick = (mask >> c) & 1;
      const auto& arcs = comps[c];
      for (size_t i = 0; i < arcs.size(); ++i) {
        if (static_cast<int>(i & 1) == pick) a[arcs[i].first] = arcs[i].second;
        else b[arcs[i].first] = arcs[i].second;
      }
    }
    if (single_cycle(a) && single_cycle(b)) return true;
  }
  return false;
}

bool decompose(int P, uint64_t seed, std::vector<int>& table) {
  table.clear();
  if (P <= 1) return true;
  if (P == 4 || P == 6 || P > 64) return false;
  const uint64_t all = (P == 64) ? ~0ull : (bit(P) - 1);
  Rng rng(seed ^ (0xA24BAED4963EE407ull * static_cast<uint64_t>(P)));
  for (int attempt = 0; attempt < 2000; ++attempt) {
    std::vector<uint64_t> out(P), in(P);
    for (int u = 0; u < P; ++u) out[u] = in[u] = all & ~bit(u);
    std::vector<std::vector<int>> cycles;
    bool ok = true;
    while (ok) {
      const int k = P - 1 - static_cast<int>(cycles.size());  // current degree
      if (k == 0) break;
      if (k == 1) {  // only possible for P == 2
        std::vector<int> s(P);
        for (int u = 0; u < P; ++u) s[u] = __builtin_ctzll(out[u]);
        if (!single_cycle(s)) { ok = false; break; }
        cycles.push_back(s);
        break;
      }
      if (k == 2) {
        std::vector<int> a, b;
        if (!split_two(P, out.data(), a, b)) { ok = false; break; }
        cycles.push_back(a);
        cycles.push_back(b);
        break;
      }
      // k >= 3: draw a Hamiltonian cycle; at k == 3 keep drawing until the
      // 2-regular remainder splits.
      const int tries = (k == 3) ? 400 : 1;
      bool got = false;
      for (int t = 0; t < tries && !got; ++t) {
        HamSearch hs{P, out.data(), in.data(), &rng, 200000, {}};
        std::vector<int> s;
        if (!hs.run(s)) continue;
        if (k == 3) {
          std::vector<uint64_t> o2 = out;
          for (int u = 0; u < P; ++u) o2[u] &= ~bit(s[u]);
          std::vector<int> a, b;
          if (!split_two(P, o2.data(), a, b)) continue;
        }
        for (int u = 0; u < P; ++u) {
          out[u] &= ~bit(s[u]);
          in[s[u]] &= ~bit(u);
        }
        cycles.push_back(s);
        got = true;
      }
      if (!got) ok = false;
    }
    if (ok && static_cast<int>(cycles.size()) == P - 1) {
      table.resize(static_cast<size_t>(P - 1) * P);
      for (int c = 0; c < P - 1; ++c)
        for (int u = 0; u < P; ++u) table[static_cast<size_t>(c) * P + u] = cycles[c][u];
      return true;
    }
  }
  return false;
}

std::mutex g_cache_mu;
std::map<std::pair<int, uint64_t>, std::vector<int>> g_cache;

bool cached_decomposition(int P, uint64_t seed, std::vector<int>& table) {
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    auto it = g_cache.find({P, seed});
    if (it != g_cache.end()) { table = it->second; return true; }
  }
  if (!decompose(P, seed, table)) return false;
  std::lock_guard<std::mutex> lk(g_cache_mu);
  g_cache[{P, seed}] = table;
  return true;
}

void split_bounds(int n, int parts, int idx, int* b, int* e) {
  const int base = n / parts, extra = n % parts;
  *b = idx * base + std::min(idx, extra);
  *e = *b + base + (idx < extra ? 1 : 0);
}

struct Docs {
  const int32_t* cu;
  int nd;
  int doc_of(int t) const {
    int lo = 0, hi = nd - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
  // True if some query in [qa,qb) may attend some key in [ka,kb).
  bool any_valid(int qa, int qb, int ka, int kb, bool causal) const {
    if (qa >= qb || ka >= kb) return false;
    if (causal && ka > qb - 1) return false;
    for (int D = doc_of(qa); D < nd && cu[D] < qb; ++D) {
      const int r1 = std::min(qb, cu[D + 1]);
      const int c0 = std::max(ka, cu[D]), c1 = std::min(kb, cu[D + 1]);
      if (c0 >= c1) continue;
      if (!causal || c0 <= r1 - 1) return true;
    }
    return false;
  }
  int flags(int qa, int qb, int ka, int kb, bool causal) const {
    int f = 0;
    if (causal && kb - 1 > qa) f |= SP_ITEM_CAUSAL_EDGE;
    const int lo = std::min(qa, ka), hi = std::max(qb, kb) - 1;
    if (doc_of(lo) != doc_of(hi)) f |= SP_ITEM_DOC_EDGE;
    return f;
  }
};

bool valid_cu(const int32_t* cu, int nd, int T) {
  if (!cu || nd < 1 || cu[0] != 0 || cu[nd] != T) return false;
  for (int i = 0; i < nd; ++i)
    if (cu[i + 1] <= cu[i]) return false;
  return true;
}

}  // namespace

extern "C" {

const char* sp_status_string(sp_status s) {
  switch (s) {
    case SP_OK: return "SP_OK";
    case SP_ERR_INVALID_ARG: return "SP_ERR_INVALID_ARG";
    case SP_ERR_UNSUPPORTED: return "SP_ERR_UNSUPPORTED";
    case SP_ERR_BUFFER_TOO_SMALL: return "SP_ERR_BUFFER_TOO_SMALL";
    case SP_ERR_CUDA: return "SP_ERR_CUDA";
    case SP_ERR_TIMEOUT: return "SP_ERR_TIMEOUT";
    case SP_ERR_INTERNAL: return "SP_ERR_INTERNAL";
  }
  return "SP_ERR_UNKNOWN";
}

sp_status sp_tasp_cycles(int32_t P, uint64_t seed, int32_t* out_succ) {
  if (P < 1) return SP_ERR_INVALID_ARG;
  if (P == 4 || P == 6 || P > 64) return SP_ERR_UNSUPPORTED;
  if (P == 1) return SP_OK;
  if (!out_succ) return SP_ERR_INVALID_ARG;
  std::vector<int> table;
  if (!cached_decomposition(P, seed, table)) return SP_ERR_INTERNAL;
  for (size_t i = 0; i < table.size(); ++i) out_succ[i] = table[i];
  return SP_OK;
}

sp_status sp_chunk_bounds(int32_t mode, int32_t P, int32_t T, const int32_t* cu, int32_t ndocs,
                          int32_t causal_i, int32_t* out) {
  if (!out || P < 1 || T < 0) return SP_ERR_INVALID_ARG;
  if (mode != SP_CHUNK_EQUAL && mode != SP_CHUNK_BALANCED && mode != SP_CHUNK_BALANCED_DOC)
    return SP_ERR_INVALID_ARG;
  if (T == 0) {
    for (int r = 0; r <= P; ++r) out[r] = 0;
    return SP_OK;
  }
  if (!valid_cu(cu, ndocs, T)) return SP_ERR_INVALID_ARG;
  if (mode == SP_CHUNK_EQUAL) {
    for (int r = 0; r < P; ++r) {
      int b, e;
      split_bounds(T, P, r, &b, &e);
      out[r] = b;
    }
    out[P] = T;
    return SP_OK;
  }
  const bool causal = causal_i != 0;
  // Work of the first m rows of a document of length L (closed form per document).
  auto doc_work = [&](int64_t m, int64_t L) { return causal ? m * (m + 1) / 2 : m * L; };
  int64_t W = 0;
  for (int d = 0; d < ndocs; ++d) W += doc_work(cu[d + 1] - cu[d], cu[d + 1] - cu[d]);
  out[0] = 0;
  int d = 0;
  int64_t before = 0;  // work of the documents before d
  for (int r = 1; r < P; ++r) {
    // Smallest t with P * W(t) >= r * W: find the document, then the row in it.
    const __int128 target = static_cast<__int128>(r) * W;
    while (d < ndocs) {
      const int64_t L = cu[d + 1] - cu[d];
      if (static_cast<__int128>(P) * (before + doc_work(L, L)) >= target) break;
      before += doc_work(L, L);
      ++d;
    }
    if (d >= ndocs) {
      out[r] = T;
      continue;
    }
    const int64_t L = cu[d + 1] - cu[d];
    auto ok = [&](int64_t m) { return static_cast<__int128>(P) * (before + doc_work(m, L)) >= target; };
    // Initial guess, then exact correction with integer checks.
    const double need = (static_cast<double>(target) / P) - static_cast<double>(before);
    int64_t m = causal ? static_cast<int64_t>(std::ceil((std::sqrt(1.0 + 8.0 * std::max(need, 0.0)) - 1.0) / 2.0))
                       : static_cast<int64_t>(std::ceil(std::max(need, 0.0) / static_cast<double>(L)));
    m = std::min<int64_t>(std::max<int64_t>(m, 0), L);
    while (m > 0 && ok(m - 1)) --m;
    while (m < L && !ok(m)) ++m;
    out[r] = cu[d] + static_cast<int32_t>(m);
  }
  out[P] = T;
  for (int r = 1; r <= P; ++r) out[r] = std::max(out[r], out[r - 1]);
  if (mode == SP_CHUNK_BALANCED_DOC && ndocs > 1) {
    // Work before each document start, and W(t) for any t.
    std::vector<int64_t> Wd(static_cast<size_t>(ndocs) + 1, 0);
    for (int x = 0; x < ndocs; ++x) Wd[x + 1] = Wd[x] + doc_work(cu[x + 1] - cu[x], cu[x + 1] - cu[x]);
    auto work_at = [&](int t) {
      const int x = static_cast<int>(std::upper_bound(cu, cu + ndocs + 1, t) - cu) - 1;
      if (x >= ndocs) return Wd[ndocs];
      return Wd[x] + doc_work(t - cu[x], cu[x + 1] - cu[x]);
    };
    for (int r = 1; r < P; ++r) {
      // The document start (cu[1 .. ndocs-1]) nearest in work to bound r: one
      // of the two around it, the earlier on a tie.
      const int64_t wb = work_at(out[r]);
      const int32_t* hi = std::lower_bound(cu + 1, cu + ndocs, out[r]);
      int best = -1;
      int64_t bdist = 0;
      for (const int32_t* c : {hi - 1, hi}) {
        if (c < cu + 1 || c >= cu + ndocs) continue;
        const int64_t dist = std::llabs(Wd[c - cu] - wb);
        if (best < 0 || dist < bdist) {
          best = *c;
          bdist = dist;
        }
      }
      if (best >= 0 && static_cast<__int128>(bdist) * 16 * P <= W && best > out[r - 1]) out[r] = best;
      else out[r] = std::max(out[r], out[r - 1]);
    }
  }
  return SP_OK;
}

sp_status sp_schedule_build(sp_sched_kind kind, int32_t P, int32_t T, const int32_t* cu,
                            int32_t ndocs, int32_t causal_i, uint64_t seed, sp_item* out,
                            int64_t* inout_n) {
  return sp_schedule_build_chunked(kind, P, T, cu, ndocs, causal_i, seed, nullptr, out, inout_n);
}

sp_status sp_schedule_build_chunked(sp_sched_kind kind, int32_t P, int32_t T, const int32_t* cu,
                                    int32_t ndocs, int32_t causal_i, uint64_t seed,
                                    const int32_t* bounds, sp_item* out, int64_t* inout_n) {
  if (!inout_n || P < 1 || T < 0) return SP_ERR_INVALID_ARG;
  if (kind != SP_SCHED_RING && kind != SP_SCHED_ZIGZAG && kind != SP_SCHED_TASP)
    return SP_ERR_INVALID_ARG;
  if (bounds && kind == SP_SCHED_ZIGZAG) return SP_ERR_UNSUPPORTED;
  if (bounds) {
    if (bounds[0] != 0 || bounds[P] != T) return SP_ERR_INVALID_ARG;
    for (int r = 0; r < P; ++r)
      if (bounds[r + 1] < bounds[r]) return SP_ERR_INVALID_ARG;
  }
  // Chunk x of the RING / TASP split.
  auto chunk = [&](int x, int* b, int* e) {
    if (bounds) {
      *b = bounds[x];
      *e = bounds[x + 1];
    } else {
      split_bounds(T, P, x, b, e);
    }
  };
  if (T == 0) {
    if (ndocs != 0 || (cu && cu[0] != 0)) return SP_ERR_INVALID_ARG;
    *inout_n = 0;
    return SP_OK;
  }
  if (!valid_cu(cu, ndocs, T)) return SP_ERR_INVALID_ARG;
  if (kind == SP_SCHED_ZIGZAG && (T % (2 * P)) != 0) return SP_ERR_UNSUPPORTED;
  if (kind == SP_SCHED_TASP && (P == 4 || P == 6 || P > 64)) return SP_ERR_UNSUPPORTED;
  const bool causal = causal_i != 0;
  Docs docs{cu, ndocs};

  std::vector<int> succ;
  std::vector<int> pred;
  if (kind == SP_SCHED_TASP && P > 1) {
    if (!cached_decomposition(P, seed, succ)) return SP_ERR_INTERNAL;
    pred.assign(succ.size(), 0);
    for (int c = 0; c < P - 1; ++c)
      for (int u = 0; u < P; ++u)
        pred[static_cast<size_t>(c) * P + succ[static_cast<size_t>(c) * P + u]] = u;
  }

  std::vector<sp_item> items;
  auto emit = [&](int r, int s, int c, int qa, int qb, int ka, int kb) {
    if (!docs.any_valid(qa, qb, ka, kb, causal)) return;
    sp_item it{r, s, c, qa, qb, ka, kb, docs.flags(qa, qb, ka, kb, causal)};
    items.push_back(it);
  };

  for (int r = 0; r < P; ++r) {
    if (kind == SP_SCHED_RING) {
      int qa, qb;
      chunk(r, &qa, &qb);
      for (int s = 0; s < P; ++s) {
        int ka, kb;
        chunk(((r - s) % P + P) % P, &ka, &kb);
        emit(r, s, 0, qa, qb, ka, kb);
      }
    } else if (kind == SP_SCHED_ZIGZAG) {
      const int c = T / (2 * P);
      const int mine[2] = {r, 2 * P - 1 - r};
      for (int a = 0; a < 2; ++a)
        for (int s = 0; s < P; ++s) {
          const int src = ((r - s) % P + P) % P;
          const int held[2] = {src, 2 * P - 1 - src};
          for (int b = 0; b < 2; ++b)
            emit(r, s, 0, mine[a] * c, (mine[a] + 1) * c, held[b] * c, (held[b] + 1) * c);
        }
    } else {
      int qa, qb;
      chunk(r, &qa, &qb);
      emit(r, 0, 0, qa, qb, qa, qb);
      for (int t = 1; t < P; ++t)
        for (int c = 0; c < P - 1; ++c) {
          int src = r;
          for (int h = 0; h < t; ++h) src = pred[static_cast<size_t>(c) * P + src];
          int cb, ce, pb, pe;
          chunk(src, &cb, &ce);
          split_bounds(ce - cb, P - 1, c, &pb, &pe);
          emit(r, t, c, qa, qb, cb + pb, cb + pe);
        }
    }
  }

  const int64_t n = static_cast<int64_t>(items.size());
  if (!out) {
    *inout_n = n;
    return SP_OK;
  }
  if (*inout_n < n) {
    *inout_n = n;
    return SP_ERR_BUFFER_TOO_SMALL;
  }
  if (n) std::memcpy(out, items.data(), sizeof(sp_item) * static_cast<size_t>(n));
  *inout_n = n;
  return SP_OK;
}

sp_status sp_schedule_build_hier(sp_sched_kind inter_kind, int32_t R, int32_t U, int32_t T,
                                 const int32_t* cu, int32_t ndocs, int32_t causal_i, uint64_t seed,
                                 int32_t Hq, const int32_t* bounds, sp_item* out, int32_t* out_heads,
                                 int64_t* inout_n) {
  if (!inout_n || R < 1 || U < 1 || Hq < 1 || Hq % U != 0 || T < 0) return SP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(R) * U > (1 << 20)) return SP_ERR_INVALID_ARG;
  // The Inter-SP schedule over the R groups.
  int64_t n = 0;
  sp_status st = sp_schedule_build_chunked(inter_kind, R, T, cu, ndocs, causal_i, seed, bounds, nullptr, &n);
  if (st != SP_OK) return st;
  std::vector<sp_item> inter(static_cast<size_t>(n));
  if (n) {
    st = sp_schedule_build_chunked(inter_kind, R, T, cu, ndocs, causal_i, seed, bounds, inter.data(), &n);
    if (st != SP_OK) return st;
  }
  const int64_t total = n * U;
  if (!out) {
    *inout_n = total;
    return SP_OK;
  }
  if (!out_heads) return SP_ERR_INVALID_ARG;
  if (*inout_n < total) {
    *inout_n = total;
    return SP_ERR_BUFFER_TOO_SMALL;
  }
  // Rank g*U + u: group g's items, query heads [u Hq/U, (u+1) Hq/U).
  const int hs = Hq / U;
  int64_t w = 0;
  size_t x = 0;
  for (int g = 0; g < R; ++g) {
    const size_t x0 = x;
    while (x < inter.size() && inter[x].rank == g) ++x;
    for (int u = 0; u < U; ++u)
      for (size_t y = x0; y < x; ++y) {
        sp_item it = inter[y];
        it.rank = g * U + u;
        out[w] = it;
        out_heads[2 * w] = u * hs;
        out_heads[2 * w + 1] = (u + 1) * hs;
        ++w;
      }
  }
  *inout_n = w;
  return SP_OK;
}

sp_status sp_schedule_split_documents(const sp_item* items, const int32_t* heads, int64_t n,
                                      const int32_t* cu, int32_t ndocs, int32_t causal_i,
                                      sp_item* out, int32_t* out_heads, int64_t* inout_n) {
  if (!inout_n || n < 0 || (n > 0 && !items) || ndocs < 1 || !cu) return SP_ERR_INVALID_ARG;
  const int T = cu[ndocs];
  if (!valid_cu(cu, ndocs, T)) return SP_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    const sp_item& it = items[i];
    if (it.q_begin < 0 || it.q_begin >= it.q_end || it.q_end > T || it.kv_begin < 0 ||
        it.kv_begin >= it.kv_end || it.kv_end > T)
      return SP_ERR_INVALID_ARG;
  }
  const bool causal = causal_i != 0;
  Docs docs{cu, ndocs};
  // A run is a maximal stretch of items sharing rank, Q range and head range
  // (one group of sp_packed_attention). Its pieces go out document by
  // document in token order, each document's pieces in input order.
  std::vector<sp_item> res;
  std::vector<int32_t> res_heads;
  std::vector<std::pair<int, int64_t>> pieces;  // (document, input index)
  auto same_run = [&](int64_t a, int64_t b) {
    return items[a].rank == items[b].rank && items[a].q_begin == items[b].q_begin &&
           items[a].q_end == items[b].q_end &&
           (!heads || (heads[2 * a] == heads[2 * b] && heads[2 * a + 1] == heads[2 * b + 1]));
  };
  for (int64_t r0 = 0; r0 < n;) {
    int64_t r1 = r0 + 1;
    while (r1 < n && same_run(r0, r1)) ++r1;
    pieces.clear();
    for (int64_t i = r0; i < r1; ++i) {
      const sp_item& it = items[i];
      const int d0 = docs.doc_of(std::max(it.q_begin, it.kv_begin));
      const int d1 = docs.doc_of(std::min(it.q_end, it.kv_end) - 1);
      for (int d = d0; d <= d1; ++d) pieces.emplace_back(d, i);
    }
    std::stable_sort(pieces.begin(), pieces.end(),
                     [](const std::pair<int, int64_t>& a, const std::pair<int, int64_t>& b) {
                       return a.first < b.first;
                     });
    for (const auto& pc : pieces) {
      const sp_item& it = items[pc.second];
      const int ds = cu[pc.first], de = cu[pc.first + 1];
      const int qa = std::max(it.q_begin, ds), qb = std::min(it.q_end, de);
      const int ka = std::max(it.kv_begin, ds), kb = std::min(it.kv_end, de);
      if (!docs.any_valid(qa, qb, ka, kb, causal)) continue;
      res.push_back(sp_item{it.rank, it.step, it.cycle, qa, qb, ka, kb, docs.flags(qa, qb, ka, kb, causal)});
      if (heads) {
        res_heads.push_back(heads[2 * pc.second]);
        res_heads.push_back(heads[2 * pc.second + 1]);
      }
    }
    r0 = r1;
  }
  const int64_t m = static_cast<int64_t>(res.size());
  if (!out) {
    *inout_n = m;
    return SP_OK;
  }
  if (heads && !out_heads) return SP_ERR_INVALID_ARG;
  if (*inout_n < m) {
    *inout_n = m;
    return SP_ERR_BUFFER_TOO_SMALL;
  }
  if (m) std::memcpy(out, res.data(), sizeof(sp_item) * static_cast<size_t>(m));
  if (heads && m) std::memcpy(out_heads, res_heads.data(), sizeof(int32_t) * 2 * static_cast<size_t>(m));
  *inout_n = m;
  return SP_OK;
}

}  // extern "C"

extern "C" sp_status sp_schedule_link_bytes(sp_sched_kind kind, int32_t P, int32_t T,
                                            const int32_t* cu, int32_t ndocs, int32_t causal_i,
                                            uint64_t seed, int64_t bytes_per_token,
                                            int32_t needed_only, int64_t* out) {
  if (P < 1 || T < 1 || bytes_per_token < 0 || (P > 1 && !out)) return SP_ERR_INVALID_ARG;
  if (kind != SP_SCHED_RING && kind != SP_SCHED_ZIGZAG && kind != SP_SCHED_TASP)
    return SP_ERR_INVALID_ARG;
  if (!valid_cu(cu, ndocs, T)) return SP_ERR_INVALID_ARG;
  if (kind == SP_SCHED_ZIGZAG && (T % (2 * P)) != 0) return SP_ERR_UNSUPPORTED;
  if (kind == SP_SCHED_TASP && (P == 4 || P == 6 || P > 64)) return SP_ERR_UNSUPPORTED;
  if (P == 1) return SP_OK;  // nothing moves
  const bool causal = causal_i != 0;
  Docs docs{cu, ndocs};
  const size_t PP = static_cast<size_t>(P) * P;
  for (size_t i = 0; i < static_cast<size_t>(P - 1) * PP; ++i) out[i] = 0;

  // Q ranges of each rank.
  std::vector<std::vector<std::pair<int, int>>> own(P);
  for (int r = 0; r < P; ++r) {
    if (kind == SP_SCHED_ZIGZAG) {
      const int c = T / (2 * P);
      own[r].push_back({r * c, (r + 1) * c});
      own[r].push_back({(2 * P - 1 - r) * c, (2 * P - r) * c});
    } else {
      int a, b;
      split_bounds(T, P, r, &a, &b);
      own[r].push_back({a, b});
    }
  }
  auto needs = [&](int r, int ka, int kb) {
    for (const auto& q : own[r])
      if (docs.any_valid(q.first, q.second, ka, kb, causal)) return true;
    return false;
  };
  // One block of keys [ka, kb) travelling along a ring whose successor is
  // next(): it starts at rank `origin` and reaches the rank h hops downstream
  // in iteration h (h = 1 .. P-1).
  auto route = [&](int origin, int ka, int kb, auto&& next) {
    if (kb <= ka) return;
    std::vector<int> path(P);
    path[0] = origin;
    for (int h = 1; h < P; ++h) path[h] = next(path[h - 1]);
    // last hop whose receiver (or someone after it) still needs the block
    int last = P - 1;
    if (needed_only) {
      last = 0;
      for (int h = P - 1; h >= 1; --h)
        if (needs(path[h], ka, kb)) { last = h; break; }
    }
    const int64_t bytes = static_cast<int64_t>(kb - ka) * bytes_per_token;
    for (int h = 1; h <= last; ++h)
      out[static_cast<size_t>(h - 1) * PP + static_cast<size_t>(path[h - 1]) * P + path[h]] += bytes;
  };

  if (kind == SP_SCHED_RING || kind == SP_SCHED_ZIGZAG) {
    auto next = [&](int r) { return (r + 1) % P; };
    for (int x = 0; x < P; ++x) {
      if (kind == SP_SCHED_RING) {
        int a, b;
        split_bounds(T, P, x, &a, &b);
        route(x, a, b, next);
      } else {
        for (const auto& q : own[x]) route(x, q.first, q.second, next);
      }
    }
    return SP_OK;
  }
  std::vector<int> succ;
  if (!cached_decomposition(P, seed, succ)) return SP_ERR_INTERNAL;
  for (int c = 0; c < P - 1; ++c) {
    auto next = [&](int r) { return succ[static_cast<size_t>(c) * P + r]; };
    for (int x = 0; x < P; ++x) {
      int cb, ce, pb, pe;
      split_bounds(T, P, x, &cb, &ce);
      split_bounds(ce - cb, P - 1, c, &pb, &pe);
      route(x, cb + pb, cb + pe, next);
    }
  }
  return SP_OK;
}

extern "C" sp_status sp_schedule_link_bytes_hier(sp_sched_kind inter_kind, int32_t R, int32_t U, int32_t T,
                                                 const int32_t* cu, int32_t ndocs, int32_t causal_i,
                                                 uint64_t seed, int32_t Hq, int32_t Hkv, int32_t d,
                                                 int32_t elem_bytes, int32_t needed_only, int64_t* intra,
                                                 int64_t* inter) {
  if (R < 1 || U < 1 || T < 1 || Hq < 1 || Hkv < 1 || d < 1 || elem_bytes < 1) return SP_ERR_INVALID_ARG;
  if (Hq % U != 0 || Hq % Hkv != 0) return SP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(R) * U > 4096) return SP_ERR_INVALID_ARG;
  const int P = R * U, hs = Hq / U, G = Hq / Hkv;
  if (!((hs >= G && hs % G == 0) || (hs < G && G % hs == 0))) return SP_ERR_UNSUPPORTED;
  if (!valid_cu(cu, ndocs, T)) return SP_ERR_INVALID_ARG;
  if (!intra || (R > 1 && !inter)) return SP_ERR_INVALID_ARG;
  if (inter_kind == SP_SCHED_ZIGZAG && T % (2 * R) != 0) return SP_ERR_UNSUPPORTED;
  const int kvs = hs >= G ? hs / G : 1;  // key/value heads one head slice needs
  const int64_t eb = elem_bytes;
  const size_t PP = static_cast<size_t>(P) * P;
  for (size_t i = 0; i < PP; ++i) intra[i] = 0;
  // Intra-SP all-to-all: rank g*U+u holds the u-th of U equal parts of group
  // g's tokens (all heads); it sends Q of query slice u' and K, V of the
  // key/value heads slice u' needs to rank g*U+u', and gets O of slice u' for
  // its own tokens back.
  for (int g = 0; g < R; ++g) {
    int gb, ge;
    if (inter_kind == SP_SCHED_ZIGZAG) {
      gb = 0;
      ge = 2 * (T / (2 * R));
    } else {
      split_bounds(T, R, g, &gb, &ge);
    }
    const int n_g = ge - gb;
    for (int u = 0; u < U; ++u) {
      int sb_, se_;
      split_bounds(n_g, U, u, &sb_, &se_);
      const int64_t n = se_ - sb_;
      for (int v = 0; v < U; ++v) {
        if (v == u) continue;
        intra[static_cast<size_t>(g * U + u) * P + (g * U + v)] += n * (hs + 2 * kvs) * d * eb;
        intra[static_cast<size_t>(g * U + v) * P + (g * U + u)] += n * hs * d * eb;
      }
    }
  }
  if (R == 1) return SP_OK;
  // Inter-SP: the R-group schedule moves, for every head slice separately,
  // the key/value heads of that slice between the ranks of that slice.
  std::vector<int64_t> grp(static_cast<size_t>(R - 1) * R * R);
  const sp_status st = sp_schedule_link_bytes(inter_kind, R, T, cu, ndocs, causal_i, seed,
                                              2 * kvs * static_cast<int64_t>(d) * eb, needed_only, grp.data());
  if (st != SP_OK) return st;
  for (size_t i = 0; i < static_cast<size_t>(R - 1) * PP; ++i) inter[i] = 0;
  for (int t = 0; t < R - 1; ++t)
    for (int a = 0; a < R; ++a)
      for (int b = 0; b < R; ++b) {
        const int64_t x = grp[static_cast<size_t>(t) * R * R + static_cast<size_t>(a) * R + b];
        if (!x) continue;
        for (int u = 0; u < U; ++u)
          inter[static_cast<size_t>(t) * PP + static_cast<size_t>(a * U + u) * P + (b * U + u)] = x;
      }
  return SP_OK;
}
