"""Planted mistakes in the oracle are caught by its pins.

Each mutant is a copy of oracle/oracle.cpp with one plausible mistake planted
in it: a mask off by one, the document start ignored, a wrong GQA head map, a
dropped scale or maximum, a transposed operand, a wrong merge weight, a wrong
sign, term or operand in a gradient; in the schedule closed forms and checks,
a reversed ring order, another zigzag layout, the remainder tokens given to
the last pieces, a check dropped or weakened, the TASP source walked the wrong
way round the cycle. Each copy is compiled on the CPU into a temporary
library. Every parameterisation of the oracle's pin tests then runs with the
oracle module pointed at that library, and at least one of them must fail:
all of test_oracle_pins.py, test_oracle_backward_pins.py and
test_oracle_schedule_pins.py, and the test_oracle_* functions of
test_chunking.py, test_comm_model.py and test_hier_schedule.py (these call
the oracle only, never the product). Mistakes are also planted in the chunk bounds (a balance bound
off by one, a causal row's work off by one, the document-snap threshold) and
in the communication model (the ring's sender, the source walked forward, the
needed-only look-ahead cut short, a TASP piece counted as a whole chunk), and
in the two-level check and model (a transposed rank layout, a wrong
renumbering, the head range's end unchecked, the attention output sent the
wrong way, another key/value-head map, K without V between groups).
The unmodified oracle passes the same list (the control), so a failure means
the pins caught the mistake, not that the harness broke."""
import contextlib
import ctypes
import itertools
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_chunking
import test_comm_model
import test_hier_schedule
import test_oracle_backward_pins
import test_oracle_pins
import test_oracle_schedule_pins

# Modules of oracle pins, and the prefix of their test functions that run the
# oracle alone (the chunking and communication modules also test the product).
PIN_MODULES = [(test_oracle_pins, "test_"), (test_oracle_backward_pins, "test_"),
               (test_oracle_schedule_pins, "test_"), (test_chunking, "test_oracle_"),
               (test_comm_model, "test_oracle_"), (test_hier_schedule, "test_oracle_")]

# name -> (text in oracle.cpp, replacement); each text occurs exactly once.
MUTANTS = {
    "causal_mask_excludes_diagonal": ("      if (causal) j1 = std::min(j1, i + 1);\n      double* o_row",
                                      "      if (causal) j1 = std::min(j1, i);\n      double* o_row"),
    "document_start_ignored": ("      int j0 = std::max(cu[D], kv_begin);",
                               "      int j0 = std::max(0, kv_begin);"),
    "gqa_head_map_interleaved": ("      const int g = h / G;\n      // V(i)",
                                 "      const int g = h % Hkv;\n      // V(i)"),
    "scale_dropped": ("        s[j - j0] = dot * scale;\n        m = std::max(m, s[j - j0]);\n      }\n      double sum",
                      "        s[j - j0] = dot;\n        m = std::max(m, s[j - j0]);\n      }\n      double sum"),
    "lse_without_maximum": ("      const double lse = m + std::log(sum);\n      std::fill(acc",
                            "      const double lse = std::log(sum);\n      std::fill(acc"),
    "values_read_from_keys": ("        for (int c = 0; c < d; ++c) acc[c] += w * widen(v, dtype, vb + c);",
                              "        for (int c = 0; c < d; ++c) acc[c] += w * widen(k, dtype, vb + c);"),
    "partial_range_end_inclusive": ("      int j1 = std::min(cu[D + 1], kv_end);",
                                    "      int j1 = std::min(cu[D + 1], kv_end + 1);"),
    "row_without_keys_gets_lse_zero": ("        lse_out[static_cast<size_t>(r) * Hq + h] = NEG_INF;\n        continue;",
                                       "        lse_out[static_cast<size_t>(r) * Hq + h] = 0.0;\n        continue;"),
    "merge_weight_offset": ("    const double wa = std::exp(a - L), wb = std::exp(b - L);",
                            "    const double wa = std::exp(a - M), wb = std::exp(b - L);"),
    "ds_sign_flipped": ("          const double ds = pij * (dp - Di);",
                        "          const double ds = pij * (Di - dp);"),
    "ds_without_rowdot": ("          const double ds = pij * (dp - Di);",
                          "          const double ds = pij * dp;"),
    "dk_from_output_gradient": ("            dk_out[kb + c] += scale * ds * qi[c];",
                                "            dk_out[kb + c] += scale * ds * doi[c];"),
    "dq_without_scale": ("            dq_out[qb + c] += scale * ds * widen(k, dtype, kb + c);",
                         "            dq_out[qb + c] += ds * widen(k, dtype, kb + c);"),
    "dv_from_ds": ("            dv_out[kb + c] += pij * doi[c];",
                   "            dv_out[kb + c] += ds * doi[c];"),
    "dp_from_keys": ("          for (int c = 0; c < d; ++c) dp += doi[c] * widen(v, dtype, kb + c);",
                     "          for (int c = 0; c < d; ++c) dp += doi[c] * widen(k, dtype, kb + c);"),
    "sampled_dp_is_the_score": ("  *dp = dpd;", "  *dp = dot;"),
    "sampled_key_queries_skip_diagonal": (
        "        for (int i = causal ? j : cu[D]; i < cu[D + 1]; ++i) {\n          const RowStats& st",
        "        for (int i = causal ? j + 1 : cu[D]; i < cu[D + 1]; ++i) {\n          const RowStats& st"),
    "sampled_dq_keys_skip_diagonal": (
        "      const int j1 = causal ? std::min(cu[D + 1], i + 1) : cu[D + 1];\n      double* out = dq_rows",
        "      const int j1 = causal ? std::min(cu[D + 1], i) : cu[D + 1];\n      double* out = dq_rows"),
    "sampled_heads_of_kv_interleaved": ("      for (int h = g * G; h < (g + 1) * G; ++h)\n        for (int i = causal ? j : cu[D]",
                                        "      for (int h = g; h < Hq; h += Hkv)\n        for (int i = causal ? j : cu[D]"),
    "row_stats_D_from_queries": ("  for (int c = 0; c < d; ++c) r.D += widen(dout, dtype, qb + c) * o[c];",
                                 "  for (int c = 0; c < d; ++c) r.D += widen(q, dtype, qb + c) * o[c];"),
    "valid_pairs_causal_off_by_one": ("      const int hi = std::min(c1, i + 1);\n      if (hi > c0)",
                                      "      const int hi = std::min(c1, i);\n      if (hi > c0)"),
    # Schedules: the closed forms and the checks.
    "ring_order_reversed": ("        const int src = ((r - s) % P + P) % P;\n        int ka, kb;",
                            "        const int src = ((r + s) % P + P) % P;\n        int ka, kb;"),
    "zigzag_mirror_chunk": ("      const int mine[2] = {r, 2 * P - 1 - r};",
                            "      const int mine[2] = {r, P + r};"),
    "piece_remainder_to_last": ("  *b = idx * base + std::min(idx, extra);\n  *e = *b + base + (idx < extra ? 1 : 0);",
                                "  *b = idx * base + std::max(0, idx - (parts - extra));\n"
                                "  *e = *b + base + (idx >= parts - extra ? 1 : 0);"),
    "hamiltonian_arc_reuse_unchecked": ("      if (++cnt > 1) return 3;", "      ++cnt;"),
    "hamiltonian_revisit_unchecked": ("      if (seen[u]) return 2;\n", ""),
    "overlap_check_weakened": ("        if (ks[y].first < ks[y - 1].second) return fail(8,",
                               "        if (ks[y].first < ks[y - 1].first) return fail(8,"),
    "pruning_check_dropped": ("    if (oracle_valid_pairs(cu, ndocs, causal, qa, qb, ka, kb) == 0)\n      return fail(4,",
                              "    if (false)\n      return fail(4,"),
    "tasp_source_walks_forward": ("        for (int t = 0; t < s; ++t) src = pred[static_cast<size_t>(c) * P + src];",
                                  "        for (int t = 0; t < s; ++t) src = succ[static_cast<size_t>(c) * P + src];"),
    # Chunk bounds (load-balanced chunking).
    "chunk_balance_off_by_one": (
        "    while (t < T && static_cast<long long>(P) * W[t] < static_cast<long long>(r) * W[T]) ++t;",
        "    while (t < T && static_cast<long long>(P) * W[t] <= static_cast<long long>(r) * W[T]) ++t;"),
    "chunk_causal_work_off_by_one": ("    const long long n = causal ? (i - cu[D] + 1) : (cu[D + 1] - cu[D]);",
                                     "    const long long n = causal ? (i - cu[D]) : (cu[D + 1] - cu[D]);"),
    "chunk_snap_threshold_halved": ("      if (16LL * P * bdist <= W[T] && best > out[r - 1]) out[r] = best;",
                                    "      if (8LL * P * bdist <= W[T] && best > out[r - 1]) out[r] = best;"),
    # Communication model (bytes per link per iteration).
    "link_ring_sender_reversed": ("        const int from = (r + P - 1) % P;", "        const int from = (r + 1) % P;"),
    "link_source_walks_forward": ("        const int src_rank = ((r - t) % P + P) % P;  // whose chunk(s) arrive",
                                  "        const int src_rank = ((r + t) % P + P) % P;  // whose chunk(s) arrive"),
    "link_lookahead_short": ("          for (int k = 0; !keep && t + k <= P - 1; ++k)\n            if (wants((r + k) % P",
                             "          for (int k = 0; !keep && t + k < P - 1; ++k)\n            if (wants((r + k) % P"),
    "link_tasp_piece_as_chunk": ("                (kb - ka) * bytes_per_token;", "                (ce - cb) * bytes_per_token;"),
    # Two-level schedules: the check and the communication model.
    "hier_slice_of_rank_transposed": ("    const int u = r % U;\n    if (heads[2 * x]",
                                      "    const int u = r / U;\n    if (heads[2 * x]"),
    "hier_renumbering_wrong": ("    for (int c = 0; c < 8; ++c) slice[u].push_back(c == 0 ? r / U : it[c]);",
                               "    for (int c = 0; c < 8; ++c) slice[u].push_back(c == 0 ? r % U : it[c]);"),
    "hier_head_end_unchecked": ("    if (heads[2 * x] != u * hs || heads[2 * x + 1] != (u + 1) * hs)",
                                "    if (heads[2 * x] != u * hs)"),
    "hier_output_sent_the_wrong_way": (
        "        intra[static_cast<size_t>(g * U + v) * P + owner] += static_cast<long long>(d) * eb;    // o",
        "        intra[static_cast<size_t>(owner) * P + (g * U + v)] += static_cast<long long>(d) * eb;    // o"),
    "hier_kv_heads_interleaved": ("  for (int h = 0; h < Hq; ++h) uses[h / hs][h / G] = 1;",
                                  "  for (int h = 0; h < Hq; ++h) uses[h / hs][h % Hkv] = 1;"),
    # Packing descriptor.
    "cu_seqlens_empty_document_accepted": ("    if (cu[i + 1] <= cu[i]) return 2;", "    if (cu[i + 1] < cu[i]) return 2;"),
    "doc_of_boundary_off_by_one": ("    if (cu[mid] <= t) lo = mid; else hi = mid - 1;",
                                   "    if (cu[mid] < t) lo = mid; else hi = mid - 1;"),
    "hier_inter_bytes_k_only": (
        "    const int rc = oracle_link_bytes(kind, R, T, cu, ndocs, causal, succ, 2 * nkv * d * eb, needed_only,",
        "    const int rc = oracle_link_bytes(kind, R, T, cu, ndocs, causal, succ, nkv * d * eb, needed_only,"),
}


def _pin_calls():
    """(label, function, kwargs) for every parameterisation of every pin test."""
    calls = []
    for mod, prefix in PIN_MODULES:
        for name in sorted(dir(mod)):
            fn = getattr(mod, name)
            if not name.startswith(prefix) or not callable(fn):
                continue
            grids = []
            for mark in getattr(fn, "pytestmark", []):
                if mark.name != "parametrize":
                    continue
                names = [n.strip() for n in mark.args[0].split(",")]
                values = list(mark.args[1])
                grids.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in values])
            for combo in itertools.product(*grids) if grids else [()]:
                kw = {}
                for part in combo:
                    kw.update(part)
                calls.append((f"{mod.__name__}.{name}{kw or ''}", fn, kw))
    return calls


def _failing_pins():
    failed = []
    for label, fn, kw in _pin_calls():
        try:
            with np.errstate(all="ignore"):  # wrong arithmetic may yield inf - inf
                fn(**kw)
        except Exception:  # an assertion, or an error the wrong arithmetic provoked
            failed.append(label)
    return failed


@contextlib.contextmanager
def _oracle_library(path):
    saved = oracle._lib
    oracle._lib = oracle._bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        oracle._lib = saved


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    src = open(oracle._SRC).read()
    d = tmp_path_factory.mktemp("oracle_mutants")
    procs, libs = [], {}
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"mutation {name}: target text not found exactly once"
        cpp = os.path.join(d, f"{name}.cpp")
        with open(cpp, "w") as f:
            f.write(src.replace(old, new))
        libs[name] = os.path.join(d, f"lib{name}.so")
        procs.append(subprocess.Popen(["g++", "-O1", "-std=c++17", "-fopenmp", "-fPIC", "-shared", cpp,
                                       "-o", libs[name]]))
    for p in procs:
        assert p.wait() == 0
    return libs


def test_unmodified_oracle_passes_every_pin():
    assert len(_pin_calls()) >= 25
    assert _failing_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant_libs, name):
    with _oracle_library(mutant_libs[name]):
        failed = _failing_pins()
    print(f"{name}: caught by {len(failed)} pin(s): {failed[:4]}")
    assert failed, f"no pin caught the planted mistake {name}"
