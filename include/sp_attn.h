/*
 * libsp_attn: the per-device hot path of sequence-parallel attention
 * (Ring / Zigzag-Ring / TASP / HSAP) on one GB300, with the P sequence-parallel
 * ranks virtual.
 *
 * Sources for what is computed:
 *  - "TASP: Topology-aware Sequence Parallelism", abstract: Ring Attention
 *    splits the query into chunks, and every Q chunk must reach every KV chunk
 *    through the iterations of a Ring AllGather; TASP decomposes the complete
 *    directed graph of ranks into orthogonal (arc-disjoint) Hamiltonian rings
 *    and the AllGather of every iteration into the same number of concurrent
 *    ring transfers.
 *  - "HSAP: A Hierarchical Sequence-aware Parallelism for Hybrid-Context
 *    Generative Models", abstract: attention on hybrid-context packed
 *    sequences must be causal and must not cross documents; the computation
 *    is a sequence of partial attention steps driven by per-device
 *    instruction sequences generated ahead of time.
 *
 * Conventions shared by every call:
 *  - T packed tokens, Hq query heads, Hkv key/value heads (Hq % Hkv == 0;
 *    query head h reads key/value head h / (Hq / Hkv)), head dim d.
 *  - Q and O: [T][Hq][d] row-major; K and V: [T][Hkv][d] row-major.
 *    LSE of a full result: [Hq][T] float32, natural log.
 *  - cu_seqlens: int32 [ndocs + 1], cu[0] = 0, strictly increasing,
 *    cu[ndocs] = T. Document i is the token range [cu[i], cu[i+1]).
 *  - Mask: query i may attend key j iff both lie in the same document and,
 *    when causal, j <= i.
 *  - Softmax scale: `scale` multiplies q.k (pass 1/sqrt(d) for the usual one).
 *  - Ownership: the caller allocates and frees every buffer; the library keeps
 *    no pointer after a call returns and allocates no device memory.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).
 *    Device work is asynchronous on it. Argument errors are returned before
 *    any launch. Device-side failures (a bounded wait that ran out, an item
 *    that is out of range) set a per-device error word that
 *    sp_check_device_status() reads.
 *  - Alignment: every device pointer must be 16-byte aligned.
 */
#ifndef SP_ATTN_H
#define SP_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SP_OK = 0,
  SP_ERR_INVALID_ARG = 1,      /* a NULL pointer, a bad size, bad cu_seqlens, a misaligned pointer */
  SP_ERR_UNSUPPORTED = 2,      /* valid but not implemented here (e.g. d not 64/128, TASP with P in {4,6}) */
  SP_ERR_BUFFER_TOO_SMALL = 3, /* output count or workspace smaller than needed */
  SP_ERR_CUDA = 4,             /* a CUDA runtime call failed */
  SP_ERR_TIMEOUT = 5,          /* a device-side bounded wait ran out */
  SP_ERR_INTERNAL = 6          /* a device-side consistency check failed */
} sp_status;

typedef enum { SP_SCHED_RING = 0, SP_SCHED_ZIGZAG = 1, SP_SCHED_TASP = 2 } sp_sched_kind;

typedef enum { SP_DTYPE_BF16 = 0, SP_DTYPE_FP32 = 1 } sp_dtype;

/* One step of one virtual rank: the Q rows [q_begin, q_end) of `rank` attend
 * the keys [kv_begin, kv_end) that reached it at `step` (over Hamiltonian
 * ring `cycle` for TASP; 0 otherwise). 32 bytes, all int32. */
typedef struct {
  int32_t rank, step, cycle, q_begin, q_end, kv_begin, kv_end, flags;
} sp_item;

#define SP_ITEM_CAUSAL_EDGE 1 /* flags bit: some pair of the item is masked by causality */
#define SP_ITEM_DOC_EDGE 2    /* flags bit: some pair of the item is masked by a document boundary */

/* sp_schedule_build — host only; builds the chunk-visit schedule ("device
 * instruction sequence", HSAP abstract) of every virtual rank.
 *
 *  kind RING:   [0,T) cut into P contiguous chunks (the first T mod P get one
 *               extra token); rank r owns chunk r; at step s it holds the KV
 *               chunk of rank (r - s) mod P (TASP abstract, Ring AllGather).
 *  kind ZIGZAG: 2P equal chunks (T % 2P must be 0); rank r owns chunks r and
 *               2P-1-r; at step s it holds both chunks of rank (r - s) mod P.
 *               One item per (own chunk, held chunk) pair.
 *  kind TASP:   P chunks as RING. P-1 arc-disjoint directed Hamiltonian
 *               cycles of the complete digraph on P ranks (deterministic in
 *               `seed`, see sp_tasp_cycles); every KV chunk is cut into P-1
 *               contiguous pieces (the first n mod (P-1) get one extra token).
 *               Step 0 is the local chunk; at step t >= 1 ring c brings piece
 *               c of the chunk of the rank t hops upstream on ring c (TASP
 *               abstract: topology decomposition and primitive decomposition).
 *               P in {4, 6} has no such decomposition: SP_ERR_UNSUPPORTED.
 *               P <= 64.
 *  Sequence-aware pruning (HSAP abstract): items without a single valid
 *  (query, key) pair under the document and causal masks are left out.
 *  Order: by rank, then the rank's Q ranges in token order, then step, then
 *  cycle (TASP) or the held chunks in token order (ZIGZAG). Items that share
 *  a rank and Q range are therefore contiguous, which sp_packed_attention
 *  requires.
 *
 *  cu_seqlens_host: host int32 [ndocs + 1]. Two-call protocol: with
 *  out_items == NULL only the count is written to *inout_n_items; otherwise
 *  *inout_n_items is the capacity on input (SP_ERR_BUFFER_TOO_SMALL if short,
 *  with the needed count written back) and the count on output. */
sp_status sp_schedule_build(sp_sched_kind kind, int32_t P, int32_t total_tokens,
                            const int32_t* cu_seqlens_host, int32_t ndocs, int32_t causal,
                            uint64_t seed, sp_item* out_items, int64_t* inout_n_items);

/* Chunking policies for the P contiguous chunks of RING and TASP schedules. */
typedef enum {
  SP_CHUNK_EQUAL = 0,        /* equal token counts (the first T mod P get one more) */
  SP_CHUNK_BALANCED = 1,     /* equal attention work per chunk */
  SP_CHUNK_BALANCED_DOC = 2  /* balanced, then boundaries moved onto nearby document starts */
} sp_chunking;

/* sp_chunk_bounds — host only; chunk boundaries out_bounds[0..P] (out_bounds[0]
 * = 0, out_bounds[P] = T, non-decreasing) for the virtual ranks. Equal token
 * counts leave a causal or packed sequence's attention work unevenly spread
 * over the ranks (load balancing: "HSAP: A Hierarchical Sequence-aware
 * Parallelism for Hybrid-Context Generative Models", Methodology; workload
 * imbalance of static sequence sharding and whole-document sharding: the
 * FlashCP abstract listed on the same page).
 *  Work of query row i: n(i) = the keys it attends (causal: i - start of its
 *  document + 1; otherwise its document's length). W(t) = sum_{i<t} n(i).
 *  SP_CHUNK_EQUAL:        the RING token split.
 *  SP_CHUNK_BALANCED:     bound r (0 < r < P) = the smallest t with
 *                         P * W(t) >= r * W(T).
 *  SP_CHUNK_BALANCED_DOC: the balanced bounds, for r = 1 .. P-1 in order:
 *                         the document start nearest to bound r in work W
 *                         (the earlier on a tie) replaces it when it moves at
 *                         most W(T) / (16P) of work and lies after bound r-1;
 *                         otherwise bound r is raised to bound r-1 if below.
 *                         Fewer documents cut across ranks, each chunk within
 *                         1/8 of the balanced work (plus one row).
 *  cu_seqlens_host as sp_schedule_build. Chunks may be empty. */
sp_status sp_chunk_bounds(int32_t mode, int32_t P, int32_t total_tokens, const int32_t* cu_seqlens_host,
                          int32_t ndocs, int32_t causal, int32_t* out_bounds);

/* sp_schedule_build_chunked — sp_schedule_build for RING or TASP with the
 * chunks given by bounds[0..P] (bounds[0] = 0, bounds[P] = T, non-decreasing;
 * NULL means SP_CHUNK_EQUAL). Rank r owns [bounds[r], bounds[r+1]); the KV
 * chunks, TASP pieces and pruning follow the same rules. ZIGZAG takes only
 * NULL (SP_ERR_UNSUPPORTED otherwise); bad bounds give SP_ERR_INVALID_ARG. */
sp_status sp_schedule_build_chunked(sp_sched_kind kind, int32_t P, int32_t total_tokens,
                                    const int32_t* cu_seqlens_host, int32_t ndocs, int32_t causal,
                                    uint64_t seed, const int32_t* bounds, sp_item* out_items,
                                    int64_t* inout_n_items);

/* sp_schedule_build_hier — host only; a two-level schedule on P = R * U
 * virtual ranks ("HSAP: A Hierarchical Sequence-aware Parallelism for
 * Hybrid-Context Generative Models", abstract and Methodology: Inter-SP
 * between device groups combined with Intra-SP inside a group; the Intra-SP
 * level read as a Ulysses-style head split, DeepSpeed-Ulysses being the
 * Intra-SP scheme the page compares with).
 *  The R groups run the Inter-SP schedule `inter_kind` (RING, ZIGZAG or TASP
 *  over R group chunks, chunk bounds as sp_schedule_build_chunked, NULL for
 *  equal). Inside group g the U ranks split the query heads: rank g*U + u
 *  holds group g's whole Q chunk and the key/value chunks group g visits, for
 *  query heads [u Hq/U, (u+1) Hq/U) (Hq % U == 0). Every item of the R-group
 *  schedule appears once per u, in rank order.
 *  out_items / out_heads (int32 [n][2], the items' query-head ranges) follow
 *  the two-call protocol of sp_schedule_build (out_items == NULL: count only).
 *  Run the result with sp_packed_attention_ex; its head ranges must then
 *  cover whole groups of Hq/Hkv heads or lie inside one (Hkv % U == 0, or
 *  Hq/U divides Hq/Hkv). */
sp_status sp_schedule_build_hier(sp_sched_kind inter_kind, int32_t R, int32_t U, int32_t total_tokens,
                                 const int32_t* cu_seqlens_host, int32_t ndocs, int32_t causal,
                                 uint64_t seed, int32_t Hq, const int32_t* bounds, sp_item* out_items,
                                 int32_t* out_heads, int64_t* inout_n_items);

/* sp_schedule_split_documents — host only; cuts every item of a schedule at
 * the document boundaries of a packed sequence, so that each output item holds
 * the (query, key) pairs of one document only ("HSAP: A Hierarchical
 * Sequence-aware Parallelism for Hybrid-Context Generative Models", abstract:
 * scheduling of incomplete QKV on hybrid-context packed sequences without
 * cross-contamination; the per-document cut is this library's reading of that
 * scheduling at document granularity, not a step the page spells out).
 *  Item (Q [a,b), KV [c,d)) becomes, for every document D = [s,e) holding a
 *  valid pair of it, the item (Q [a,b) n D, KV [c,d) n D) with the same rank,
 *  step and cycle and flags recomputed for the piece (SP_ITEM_DOC_EDGE is then
 *  never set). The valid pairs covered are exactly the input's.
 *  Order: each maximal run of consecutive items sharing rank, Q range and (if
 *  heads is given) head range is replaced by its pieces, document by document
 *  in token order, each document's pieces in input order. The pieces of one run
 *  and one document share a Q range, so sp_packed_attention runs every
 *  document of a rank's chunk as a group of its own: its units walk one
 *  document's keys, and groups are started longest walk first.
 *  items: host, n_items items with 0 <= q_begin < q_end <= T and
 *  0 <= kv_begin < kv_end <= T (T = cu_seqlens_host[ndocs]), else
 *  SP_ERR_INVALID_ARG. heads: host int32 [n_items][2] query-head ranges
 *  (sp_schedule_build_hier) or NULL; out_heads receives the pieces' ranges and
 *  must be given when heads is. cu_seqlens_host as sp_schedule_build (ndocs >=
 *  1). Two-call protocol of sp_schedule_build for out_items / *inout_n_items.
 *  The cut multiplies the groups by the documents a rank's chunk spans;
 *  sp_packed_attention takes at most SP_MAX_GROUPS of them.
 *  Nothing is kept; the inputs are only read. */
sp_status sp_schedule_split_documents(const sp_item* items, const int32_t* heads, int64_t n_items,
                                      const int32_t* cu_seqlens_host, int32_t ndocs, int32_t causal,
                                      sp_item* out_items, int32_t* out_heads, int64_t* inout_n_items);

/* sp_tasp_cycles — host only. Writes the P-1 Hamiltonian cycles that TASP
 * schedules use for (P, seed) as successor tables: out_succ[c * P + u] is the
 * rank after u on ring c. out_succ must hold (P-1)*P int32. P = 1 writes
 * nothing. Same errors as the TASP schedule. Results are cached per (P, seed). */
sp_status sp_tasp_cycles(int32_t P, uint64_t seed, int32_t* out_succ);

/* sp_schedule_link_bytes — host only; the communication volume a schedule
 * implies on the virtual ranks' links ("TASP: Topology-aware Sequence
 * Parallelism", abstract: a Ring AllGather is P-1 iterations of ring transfers
 * that use only one ring of links; TASP decomposes the complete digraph into
 * P-1 Hamiltonian rings and moves one piece of every chunk on each ring in
 * every iteration).
 *  out[(t-1)*P*P + u*P + v] = bytes sent over the directed link u -> v in
 *  transfer iteration t = 1 .. P-1:
 *   RING:   rank r receives from r-1 the chunk that started at rank r-t;
 *   ZIGZAG: the same ring, carrying both chunks of rank r-t;
 *   TASP:   on ring c, rank r receives from its predecessor on c piece c of the
 *           chunk that started t hops upstream on c.
 *  A block of keys costs (kv_end - kv_begin) * bytes_per_token.
 *  needed_only != 0: a block stops travelling after the last rank on its ring
 *  that needs it (a query with a valid key in the block; sequence-aware
 *  pruning, HSAP abstract); otherwise the full AllGather is counted.
 *  out: caller-allocated int64 [(P-1)*P*P] (unused when P == 1).
 *  Errors as sp_schedule_build. */
sp_status sp_schedule_link_bytes(sp_sched_kind kind, int32_t P, int32_t total_tokens,
                                 const int32_t* cu_seqlens_host, int32_t ndocs, int32_t causal,
                                 uint64_t seed, int64_t bytes_per_token, int32_t needed_only,
                                 int64_t* out);

/* sp_schedule_link_bytes_hier — host only; communication volume of a
 * two-level schedule (sp_schedule_build_hier) on P = R * U virtual ranks,
 * inputs in `elem_bytes`-byte elements.
 *  intra[u*P + v] (int64 [P*P]): bytes over the directed link u -> v of the
 *    Intra-SP all-to-all of one attention call: rank g*U+u first holds the
 *    u-th of U equal parts of group g's tokens (all heads); it sends Q of
 *    query-head slice u' and K, V of the key/value heads slice u' needs to
 *    rank g*U+u' (u' != u), and receives O of slice u' for its tokens back.
 *    (Group chunks: the equal RING/TASP split, or the ZIGZAG pair.)
 *  inter[(t-1)*P*P + u*P + v] (int64 [(R-1)*P*P], unused for R == 1): the
 *    Inter-SP transfers per iteration t, as sp_schedule_link_bytes for the
 *    R groups, carried separately between the ranks of each head slice with
 *    that slice's key/value heads (bytes per token 2 * kv_heads * d * elem_bytes).
 *  Head slices must cover whole key/value-head groups or lie inside one
 *  (SP_ERR_UNSUPPORTED otherwise). */
sp_status sp_schedule_link_bytes_hier(sp_sched_kind inter_kind, int32_t R, int32_t U, int32_t total_tokens,
                                      const int32_t* cu_seqlens_host, int32_t ndocs, int32_t causal,
                                      uint64_t seed, int32_t Hq, int32_t Hkv, int32_t d, int32_t elem_bytes,
                                      int32_t needed_only, int64_t* intra, int64_t* inter);

/* sp_partial_attn — one partial attention step ("partial attention
 * computation", HSAP abstract; one iteration of Ring Attention, TASP abstract).
 * For every query row t in [q_begin, q_end) and head h, over the keys
 * j in [kv_begin, kv_end) that the mask allows:
 *   lse_part[h][t - q_begin] = log sum_j exp(scale * q_t.k_j)
 *   o_part[t - q_begin][h][:] = sum_j exp(scale * q_t.k_j - lse) v_j
 * A row with no allowed key gets lse = -inf and o = 0.
 *  q, k, v: device, dtype as given (bf16 runs on the tensor cores; fp32 runs on
 *           CUDA cores in fp32 for the 1e-5 tolerance).
 *  o_part: device float32 [q_end - q_begin][Hq][d]; lse_part: device float32
 *          [Hq][q_end - q_begin].
 *  cu_seqlens_dev: device int32 [ndocs + 1]. Not checked here (no set-up
 *           kernel runs): a malformed descriptor changes the masks but every
 *           access stays within the Q rows and key range given.
 *  d must be 64 or 128. An empty row range is a no-op. */
sp_status sp_partial_attn(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                          int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                          int32_t q_begin, int32_t q_end, int32_t kv_begin, int32_t kv_end,
                          const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal, float scale,
                          void* stream);

/* sp_lse_merge — folds one normalised partial into an accumulator, in place:
 * the step that combines the results of "partial attention computation"
 * (HSAP abstract) across the iterations of a Ring Attention schedule (TASP
 * abstract). The pages name no formula; the rule is the log-sum-exp merge,
 * exact for partials over disjoint key sets:
 *   M = max(L1, L2), L = M + log(exp(L1 - M) + exp(L2 - M)),
 *   O = exp(L1 - L) O1 + exp(L2 - L) O2.
 * A partial with L = -inf is the identity; two -inf stay -inf with O = 0.
 *  o_acc, o_part: device float32 [rows][Hq][d]; lse_acc, lse_part: device
 *  float32 [Hq][rows]. d % 4 == 0. Bandwidth bound: 12 bytes per O element. */
sp_status sp_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                       int32_t rows, int32_t Hq, int32_t d, void* stream);

/* Bytes of device workspace sp_packed_attention needs for n_items items. */
size_t sp_packed_attention_workspace_size(int64_t n_items);

/* sp_packed_attention — the whole schedule in one persistent launch (plus a
 * small set-up kernel): for every query row, the items of its rank and Q range
 * are visited in schedule order and their partials are merged on chip with
 * the log-sum-exp rule, so the result is exact masked attention over each
 * packed document (HSAP abstract; TASP abstract).
 *  o: device [T][Hq][d] in `dtype` (bf16 rounded to nearest even); lse: device
 *     float32 [Hq][T], natural log.
 *  items_dev: device copy of a schedule from sp_schedule_build (or any item
 *     list whose Q ranges do not overlap across groups and whose items with
 *     the same rank and Q range are contiguous); rows of [0, T) covered by no
 *     item are not written.
 *  workspace: device, at least sp_packed_attention_workspace_size(n_items)
 *     bytes, owned by the caller, reused between calls; calls that share a
 *     workspace must not overlap in time.
 *  n_items < 2^30 (SP_ERR_INVALID_ARG otherwise). The order in which a unit
 *  merges its items' partials is free (the log-sum-exp merge is associative):
 *  items that are not whole 128-key tiles long are visited in key order, and
 *  contiguous key ranges are walked as one.
 *  Checked on the device before anything is written (a failure is reported
 *  as SP_ERR_INTERNAL through sp_check_device_status, and no output is
 *  touched): cu_seqlens_dev is a packing descriptor of [0, T) (cu[0] = 0,
 *  strictly increasing, cu[ndocs] = T); every item lies in [0, T) and holds
 *  at least one (query, key) pair the masks allow under it, as a pruned
 *  schedule built from the same descriptor does (an item without one means
 *  the schedule was built for another packing); the items form at most
 *  SP_MAX_GROUPS groups (runs sharing a rank, Q range and head range) whose Q
 *  ranges do not overlap. */
#define SP_MAX_GROUPS 8192
sp_status sp_packed_attention(const void* q, const void* k, const void* v, void* o, float* lse,
                              int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                              const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal, float scale,
                              const sp_item* items_dev, int64_t n_items, void* workspace,
                              size_t workspace_bytes, void* stream);

/* sp_packed_attention_ex — sp_packed_attention over items that each cover a
 * range of query heads, as hierarchical schedules produce (an Intra-SP head
 * split under an Inter-SP ring: "HSAP: A Hierarchical Sequence-aware
 * Parallelism for Hybrid-Context Generative Models", abstract and
 * Methodology; see sp_schedule_build_hier).
 *  item_heads_dev: device int32 [n_items][2], query heads [h_begin, h_end) of
 *     each item (NULL: all heads, which is sp_packed_attention). A range must
 *     cover whole groups of Hq/Hkv query heads or lie inside one group.
 *     Items that share a rank, Q range and head range must be contiguous;
 *     the (Q range x head range) rectangles of different groups must not
 *     overlap. Violations are reported through sp_check_device_status
 *     (SP_ERR_INTERNAL, nothing written).
 *  Other arguments as sp_packed_attention; rows and heads no item covers are
 *  not written. */
sp_status sp_packed_attention_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                                 const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal,
                                 float scale, const sp_item* items_dev, const int32_t* item_heads_dev,
                                 int64_t n_items, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* sp_packed_attention_static_ws — sp_packed_attention for callers that cannot
 * allocate device memory. The pages have no counterpart to this call.
 *
 * Some callers have no way to obtain the scratch buffer sp_packed_attention
 * asks for: a plugin that is handed only its input and output pointers by a
 * host framework that owns all device memory, a binding with no CUDA
 * allocator of its own, or a serving loop that must not call cudaMalloc or
 * cudaFree (which synchronise the device) once it is running. This variant
 * takes the same arguments without the workspace and uses instead a fixed
 * scratch array of SP_STATIC_WS_BYTES compiled into the library; every GPU
 * that loads the library reserves that array until the process exits.
 *  - Limit: n_items <= SP_STATIC_WS_MAX_ITEMS; longer schedules are rejected
 *    with SP_ERR_BUFFER_TOO_SMALL before anything is launched.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - All calls on a device share the one array. The set-up kernel rewrites
 *    every word the attention kernel reads, so nothing is carried over from
 *    the previous call, but two calls whose work overlaps on the GPU (for
 *    example on two streams) race on the array: serialise them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define SP_STATIC_WS_BYTES (4u << 20)
#define SP_STATIC_WS_MAX_ITEMS 40000
sp_status sp_packed_attention_static_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                                        int32_t T, int32_t Hq, int32_t Hkv, int32_t d, sp_dtype dtype,
                                        const int32_t* cu_seqlens_dev, int32_t ndocs, int32_t causal,
                                        float scale, const sp_item* items_dev, int64_t n_items,
                                        void* stream);

/* Bytes of device workspace sp_packed_attention_backward needs: a small
 * header, two fp32 [Hq][T] row vectors and an fp32 [T][Hq][128] dQ
 * accumulator (n_items does not change it). */
size_t sp_packed_attention_backward_workspace_size(int64_t n_items, int32_t T, int32_t Hq);

/* sp_packed_attention_backward — gradients of sp_packed_attention for
 * training with the sequence-parallel schedules (HSAP abstract: training
 * throughput in tokens per GPU per second). With P_tj = exp(scale q_t.k_j -
 * LSE_t) over the keys the mask allows, D_t = dO_t . O_t, dP_tj = dO_t . v_j,
 * dS_tj = P_tj (dP_tj - D_t):
 *   dQ_t = scale sum_j dS_tj k_j,  dK_j = scale sum_t dS_tj q_t,
 *   dV_j = sum_t P_tj dO_t,
 * dK and dV of a key/value head summing over the query heads of its group.
 *  q, k, v, o, dout: device bf16 as in sp_packed_attention (o and lse are the
 *     forward's outputs for the same inputs; dout has the layout of o).
 *  lse: device float32 [Hq][T], natural log, as the forward wrote it.
 *  dq: device bf16 [T][Hq][d]; dk, dv: device bf16 [T][Hkv][d]; every element
 *     is written (keys no query attends and queries without keys get 0).
 *  items_dev: a complete schedule (every pair the mask allows exactly once,
 *     as sp_schedule_build produces). The gradients are sums over the pairs
 *     the mask allows, which for a complete schedule are the pairs its items
 *     hold; they are accumulated key tile by key tile, so the items fix only
 *     the order of the sums and are not read (n_items must still be >= 1).
 *  dK and dV are bit-reproducible from run to run; dQ is summed with fp32
 *     reductions in global memory whose order varies, so its low bits may.
 *  dtype must be SP_DTYPE_BF16 (SP_ERR_UNSUPPORTED otherwise); d is 64 or 128.
 *  workspace: device, at least sp_packed_attention_backward_workspace_size
 *     bytes, owned by the caller; calls sharing it must not overlap in time.
 *  cu_seqlens_dev is checked on the device as in sp_packed_attention; a bad
 *  one is reported as SP_ERR_INTERNAL and dq, dk, dv are not touched.
 *  Timeouts of the kernels' bounded waits are reported through
 *  sp_check_device_status. */
sp_status sp_packed_attention_backward(const void* q, const void* k, const void* v, const void* o,
                                       const void* dout, const float* lse, void* dq, void* dk,
                                       void* dv, int32_t T, int32_t Hq, int32_t Hkv, int32_t d,
                                       sp_dtype dtype, const int32_t* cu_seqlens_dev, int32_t ndocs,
                                       int32_t causal, float scale, const sp_item* items_dev,
                                       int64_t n_items, void* workspace, size_t workspace_bytes,
                                       void* stream);

/* Synchronises `stream`, reads and clears the current device's error word, and
 * returns SP_OK, SP_ERR_TIMEOUT, SP_ERR_INTERNAL, or SP_ERR_CUDA when the
 * stream itself reports a CUDA error. */
sp_status sp_check_device_status(void* stream);

/* Diagnostic: launches one block whose thread waits on a barrier that nothing
 * completes, bounded by timeout_ns of GPU time; the wait gives up, records
 * SP_ERR_TIMEOUT in the error word and the block exits normally. Checks that
 * bounded waits end and report. */
sp_status sp_selftest_bounded_wait(uint64_t timeout_ns, void* stream);

/* Human-readable name of a status code (static storage). */
const char* sp_status_string(sp_status s);

#ifdef __cplusplus
}
#endif

#endif /* SP_ATTN_H */
