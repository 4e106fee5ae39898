/*
 * libkvc -- budgeted KV-cache compaction on one GB300 (sm_103a).
 *
 * One compaction pass over a KV cache, per unit u = (sequence b, layer l,
 * KV head g), units ordered [B][L][H_kv]:
 *
 *   kvc_score                   window-attention mass of every cached token
 *                               (+ bonus, optional page max)
 *   kvc_select                  deterministic budgeted selection
 *   kvc_compact_rerotate_quant  gather kept K/V rows, re-rotate kept keys to
 *                               their new positions, quantise, store
 *   kvc_compact_rerotate_quant_ref   the same through a key reference store
 *   kvc_decode_attn             one decode-attention step over the result
 *
 * Sources, cited by page title and section:
 *   PASK     "Parser Transitions Already Reveal Structural Responsibility:
 *             KV Persistence for Structured Generation" (arXiv 2608.28276)
 *   PACE     "PACE: Keeping the Right Tokens in the KV Cache Is Not Enough
 *             for Long-Horizon LLM Agents" (arXiv 2611.10240)
 *   CommitKV "CommitKV: Lifecycle-Aware KV Cache Compression via Commit
 *             Transitions for Multi-Turn Agents" (arXiv 2608.07855)
 *
 * Conventions shared by every entry point
 *   - Every data pointer is DEVICE memory of the current CUDA device, owned
 *     by the caller, unless a call says otherwise.  The library keeps no pointer after a call returns and
 *     allocates no device memory; scratch space is the caller's workspace,
 *     sized by the matching *_workspace_bytes call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise.  Results are valid once the
 *     caller synchronises the stream.
 *   - Inputs are read-only (except `scores` under KVC_SCORE_ACCUMULATE).
 *     Outputs must not alias inputs.
 *   - Errors detectable from the arguments (null pointers, shapes, sizes,
 *     alignment, capacity) are returned before anything is launched.
 *     Conditions that depend on device data are written per unit to a
 *     `unit_status` array (KVC_UNIT_*), never by trapping the GPU.
 *   - Element layouts: bf16 = IEEE bfloat16 bits, fp16 = IEEE half bits,
 *     row-major, innermost index last.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, passed as a plain pointer. */
typedef void* kvc_stream;

/* Host-side return codes. */
typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1,  /* a null pointer, a bad shape or size         */
  KVC_ERR_UNSUPPORTED = 2,  /* a valid request the library does not handle */
  KVC_ERR_WORKSPACE = 3,    /* workspace missing or too small             */
  KVC_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed        */
  KVC_ERR_NO_DEVICE = 5     /* no usable sm_103 device                    */
} kvc_status;

/* Per-unit device status, written to unit_status[u]. */
enum {
  KVC_UNIT_OK = 0,
  KVC_UNIT_OVER_BUDGET = 1, /* forced rows alone exceed the token budget   */
  KVC_UNIT_BAD_INDEX = 2,   /* a kept index or position outside its range */
  KVC_UNIT_BAD_FLAGS = 3,   /* an item flagged both PROTECT and EXCLUDE    */
  KVC_UNIT_TIMEOUT = 4      /* a bounded device wait gave up (no progress) */
};

/* Storage actions of the (tag, layer-group) table: PASK's {R, L, H} with L
 * split into int4 and int8.  Pool index of a stored action = action - 1. */
enum { KVC_ACT_RELEASE = 0, KVC_ACT_INT4 = 1, KVC_ACT_INT8 = 2, KVC_ACT_BF16 = 3 };
enum { KVC_POOL_INT4 = 0, KVC_POOL_INT8 = 1, KVC_POOL_BF16 = 2, KVC_N_POOLS = 3 };

/* Per-token (or per-page) flag bits. */
enum { KVC_FLAG_PROTECT = 1, KVC_FLAG_EXCLUDE = 2 };

/* Quantisation modes. */
enum {
  KVC_QUANT_G32_BF16 = 0,   /* groups of 32 elements, bf16 scale per group */
  KVC_QUANT_ROW_FP16 = 1    /* one fp16 scale per row (PASK App. B.5)      */
};

/* Rotary layouts of the stored keys (PACE Sec. 3.2: re-rotation applies the
 * same rotation to the rotated dimensions only).  Split halves pair element
 * i with i + rotary_dim/2; interleaved pairs 2i with 2i + 1.  The cos / sin
 * tables hold rotary_dim / 2 columns. */
enum { KVC_ROPE_SPLIT_HALF = 0, KVC_ROPE_INTERLEAVED = 1 };

/* kvc_score flags. */
enum { KVC_SCORE_ACCUMULATE = 1 };

typedef struct {
  int32_t batch;       /* B                                        */
  int32_t n_layers;    /* L                                        */
  int32_t n_q_heads;   /* H_q, a multiple of H_kv                  */
  int32_t n_kv_heads;  /* H_kv; G = H_q / H_kv query heads per KV head */
  int32_t head_dim;    /* d: 64 or 128                             */
  int64_t n_tokens;    /* T: cached rows per unit before compaction */
} kvc_shape;

/* ------------------------------------------------------------------------
 * kvc_score -- observation-window attention mass (step a1/a2).
 *
 * PASK Eq. 1 (causal attention, softmax over K^T q / sqrt(d)); the window
 * scorer (SnapKV, described in PASK App. C.3 and CommitKV Sec. 3.1): the
 * last `window` queries of every query head score all cached keys, and the
 * softmax weights are summed over the window rows and over the G query heads
 * that share the KV head; PACE Sec. 3.1 adds an external bonus to the score.
 * Query head h reads KV head h / G.  Window row w sits at cache index
 * T - window + w and sees keys j <= T - window + w.
 *
 *   scores[u][j] = sum_{h in g} sum_w softmax_j(q_{h,w} . k_j * scale)
 *                  + bonus[b][j] (+ scores[u][j] if KVC_SCORE_ACCUMULATE)
 *   page_scores[u][p] = max_{j in page p} scores[u][j]      (page_size > 1)
 *
 * k_cache   bf16 [B][L][H_kv][T][d], keys rotated at their positions;
 *           16-byte aligned.
 * q_window  bf16 [B][L][H_q][window][d], rotated; 16-byte aligned.
 * window    W >= 1, W <= T, W * G <= 256 (W = 1 scores one decode query per
 *           head, the H2O cumulative score with KVC_SCORE_ACCUMULATE).
 * softmax_scale  <= 0 selects 1 / sqrt(d).
 * row_lse   optional fp32 [B][L][H_q][window]: the natural-log log-sum-exp
 *           of each window row's logits q_{h,w} . k_j * scale over the keys
 *           it sees, when the caller already has it (an attention kernel
 *           that produced the window's outputs returns it).  The row
 *           statistics pass is then skipped and softmax_j is formed as
 *           exp(q_{h,w} . k_j * scale - row_lse[h][w]).  NULL = computed
 *           here (two passes over the keys).
 * bonus     optional fp32 [B][T] (NULL = 0).
 * page_size 1 (no page scores) or 2, 4, 8, 16, 32 with T % page_size == 0.
 * scores    fp32 [U][T] (read too under KVC_SCORE_ACCUMULATE).
 * page_scores  fp32 [U][T / page_size]; required iff page_size > 1.
 * unit_status  optional int32 [U]; KVC_UNIT_TIMEOUT if a device wait gave
 *           up; untouched otherwise.
 * workspace >= kvc_score_workspace_bytes(shape, window) bytes, 256-byte
 *           aligned; its contents need not be initialised.
 * ---------------------------------------------------------------------- */
size_t kvc_score_workspace_bytes(const kvc_shape* shape, int32_t window);
kvc_status kvc_score(const kvc_shape* shape, const void* k_cache, const void* q_window,
                     int32_t window, float softmax_scale, const float* row_lse, const float* bonus,
                     int32_t page_size, uint32_t flags, float* scores, float* page_scores,
                     int32_t* unit_status, void* workspace, size_t workspace_bytes,
                     kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_foresight_bonus -- PACE Eq. 2 foresight bonus of every token.
 *
 * PACE Sec. 3.1: at step t a token in a span (a, b, F) of the blueprint's
 * forward-reference table, whose next reference is s* = min{s in F: s >= t},
 * receives beta = sigma (1/2 + 1/2 exp(-lambda (s* - t))); tokens with no
 * future reference receive 0 (a token in several spans takes the largest
 * bonus).  The bonus is what kvc_score adds to each token's score (pass it
 * as `bonus`), so that with sigma / 2 above every cumulative attention
 * score each referenced token outranks each unreferenced one.
 *
 * span_seq   int32 [n_spans]: the sequence b each span belongs to.
 * span_a, span_b  int64 [n_spans]: token range [a, b) (clipped to [0, T)).
 * span_next  int32 [n_spans]: s* computed by the caller; a value < step
 *            means no future reference (the span contributes nothing).
 * step       t.  sigma > 0 (PACE: 1e5), lambda >= 0 (PACE: 0.35).
 * bonus      fp32 [batch][n_tokens], overwritten.
 * ---------------------------------------------------------------------- */
kvc_status kvc_foresight_bonus(int32_t batch, int64_t n_tokens, const int32_t* span_seq,
                               const int64_t* span_a, const int64_t* span_b,
                               const int32_t* span_next, int32_t n_spans, int32_t step,
                               float sigma, float lambda, float* bonus, kvc_stream stream);

/* ------------------------------------------------------------------------
 * Selection policy.  Exactly one of budget_tokens / budget_bytes is > 0.
 *
 * Token / page mode (budget_tokens > 0): per unit keep the forced items
 * (n_sink first tokens, n_recent last tokens, PROTECT-flagged items) and
 * fill the budget with the eligible items (not forced, not EXCLUDE-flagged)
 * that rank first by (score descending, index ascending), after mapping
 * -0 to +0 and NaN to -inf.  If the forced items alone exceed the budget
 * the unit is KVC_UNIT_OVER_BUDGET and keeps nothing (CommitKV Eq. 4,
 * |I| <= B; Eq. 13, protected pages are kept).  Page mode (page_size > 1)
 * selects whole pages by page score: a page is forced if it holds a sink or
 * recent token; budget_tokens must be a multiple of page_size.  All kept
 * rows go to the bf16 pool.
 *
 * Byte mode (budget_bytes > 0): PASK's floor-constrained allocation
 * (App. B.3-B.4, Sec. 3.5).  Each token's floor action is
 * action_table[tags[b][t]][group(l)] with group(l) the layer group of
 * PASK App. A.2 generalised to n_layer_groups groups,
 * b_k = floor((k L + G - 1) / G).  Sink, recent and PROTECT tokens are
 * bf16, EXCLUDE tokens are released.  Row cost (K+V bytes): bf16 4d;
 * int8 2(d + s); int4 2(d/2 + s) with s = 2 d/32 (g32) or 2 (row mode).
 * The remainder budget_bytes - sum(floor costs) is spent by promoting to
 * bf16 the longest prefix of the (score desc, index asc) order of the
 * remaining non-bf16 tokens whose summed upgrade costs fit; a negative
 * remainder is written to floor_excess and nothing is promoted.
 *
 * renumber: 1 = kept rows get new positions 0..n_kept-1 in index order
 *           (PACE Sec. 3.2 bounded positions), 0 = positions unchanged
 *           (CommitKV Eq. 4).
 * capacity: rows per pool per unit of the output arrays; must be >=
 *           budget_tokens (token/page mode) or >= T (byte mode).
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t budget_tokens;
  int64_t budget_bytes;
  int32_t n_sink;
  int32_t n_recent;
  int32_t page_size;       /* 1 = token mode                              */
  int32_t renumber;
  int32_t capacity;
  int32_t quant_mode;      /* KVC_QUANT_*                                 */
  int32_t n_tags;          /* byte mode: rows of action_table             */
  int32_t n_layer_groups;  /* byte mode: columns of action_table          */
  const uint8_t* flags;    /* optional uint8 [B][T] (token mode) or [B][T/P] (page mode) */
  const uint8_t* tags;     /* byte mode: uint8 [B][T], each < n_tags      */
  const uint8_t* action_table; /* byte mode: uint8 [n_tags][n_layer_groups] of KVC_ACT_* */
  int32_t rope_layout;     /* KVC_ROPE_SPLIT_HALF (0) or KVC_ROPE_INTERLEAVED */
  int32_t rotary_dim;      /* rotated leading dimensions, a multiple of 16; 0 = head_dim */
} kvc_policy;

/* ------------------------------------------------------------------------
 * kvc_select -- masks and deterministic top-k / byte-budget selection
 * (steps a3/a4).
 *
 * scores       fp32 [U][T] (token and byte mode) or [U][T/P] (page mode).
 * kept_idx     int32 [KVC_N_POOLS][U][capacity]: kept token indices of each
 *              pool, ascending; entries past kept_count are not written.
 * kept_count   int32 [KVC_N_POOLS][U].
 * unit_status  int32 [U], always written (KVC_UNIT_OK or an error code;
 *              KVC_UNIT_TIMEOUT, with nothing kept, if a unit's scores did
 *              not reach shared memory within the bounded device wait).
 * floor_excess optional int64 [U] (byte mode; 0 otherwise).
 * workspace    optional: in token and page mode with more than 32,768 items
 *              per unit, a workspace of kvc_select_workspace_bytes (256-byte
 *              aligned; contents need not be initialised) lets the selection
 *              of every unit run over many CTAs; without it each unit is
 *              selected by one CTA (same result, slower).  Otherwise the
 *              size is 0 and NULL is accepted.
 * ---------------------------------------------------------------------- */
size_t kvc_select_workspace_bytes(const kvc_shape* shape, const kvc_policy* policy);
kvc_status kvc_select(const kvc_shape* shape, const kvc_policy* policy, const float* scores,
                      int32_t* kept_idx, int32_t* kept_count, int32_t* unit_status,
                      int64_t* floor_excess, void* workspace, size_t workspace_bytes,
                      kvc_stream stream);

/* ------------------------------------------------------------------------
 * Selection variants on the score buffer.
 *
 * kvc_pool_scores -- SnapKV's pooling of token scores before selection (the
 * pooling and kernel options of the SnapKV baseline in PASK's baseline
 * table): pooled[r][j] = average (KVC_SCORE_POOL_AVG) or maximum
 * (KVC_SCORE_POOL_MAX) of scores[r][j - kernel/2 .. j + kernel/2]; outside
 * [0, n_tokens) a score counts as 0 in the average (always divided by
 * `kernel`) and is ignored by the maximum.  kernel is 1, 3, 5 or 7.
 * scores, pooled: fp32 [n_rows][n_tokens], distinct buffers; n_rows <= 65535.
 *
 * kvc_shared_scores -- CommitKV Eq. 4 applies one index set I_j to the keys,
 * values and positions of every layer and head: shared[b][j] = sum over the
 * sequence's units (l, g) of scores[(b, l, g)][j], summed in unit order.
 * scores fp32 [U][T] (U = B L H_kv); shared fp32 [B][T].
 *
 * kvc_broadcast_kept -- copies the kept lists selected on the shared scores
 * (kvc_select called with a shape of B units: n_layers = n_kv_heads = 1) to
 * every unit of the sequence, ready for kvc_compact_rerotate_quant.
 * kept_idx_seq int32 [KVC_N_POOLS][B][capacity], kept_count_seq [KVC_N_POOLS][B];
 * kept_idx int32 [KVC_N_POOLS][U][capacity], kept_count [KVC_N_POOLS][U].
 * ---------------------------------------------------------------------- */
enum { KVC_SCORE_POOL_AVG = 0, KVC_SCORE_POOL_MAX = 1 };

kvc_status kvc_pool_scores(int64_t n_rows, int64_t n_tokens, const float* scores, float* pooled,
                           int32_t kernel, int32_t mode, kvc_stream stream);
kvc_status kvc_shared_scores(const kvc_shape* shape, const float* scores, float* shared,
                             kvc_stream stream);
kvc_status kvc_broadcast_kept(const kvc_shape* shape, const kvc_policy* policy,
                              const int32_t* kept_idx_seq, const int32_t* kept_count_seq,
                              int32_t* kept_idx, int32_t* kept_count, kvc_stream stream);

/* Compacted pools.  A pool's pointers may be NULL when no call will store a
 * row in it (token and page mode use only the bf16 pool). */
typedef struct {
  void* k_bf16;      /* bf16 [U][capacity][d]                                  */
  void* v_bf16;
  void* k_i8;        /* int8 codes [U][capacity][d]                            */
  void* v_i8;
  void* k_i8_scale;  /* g32: bf16 [U][capacity][d/32]; row mode: fp16 [U][capacity] */
  void* v_i8_scale;
  void* k_i4;        /* packed int4 [U][capacity][d/2]: element 2j in the low nibble */
  void* v_i4;
  void* k_i4_scale;  /* as k_i8_scale */
  void* v_i4_scale;
  int32_t* pos_out;      /* int32 [KVC_N_POOLS][U][capacity]: new position */
  int32_t* orig_pos_out; /* optional, same layout: position before compaction */
} kvc_pools;

/* ------------------------------------------------------------------------
 * kvc_compact_rerotate_quant -- gather, renumber, re-rotate, quantise,
 * store (steps a5/a6).
 *
 * CommitKV Eq. 4: the kept index set is applied to K, V and positions.
 * PACE Sec. 3.2: with renumber on, kept row i of the unit (all pools merged
 * in index order) gets position p' = its rank; its key, stored rotated at
 * p, is re-rotated by R_{p'-p} (Prop. 1), the cosine and sine of (p'-p)
 * theta_i being formed from the caller's tables by the angle-difference
 * identities and normalised to unit length.  Split-half rotary layout:
 * element i pairs with i + d/2.  Fixed fp32 order, no fused multiply-add:
 *   C = c'c + s's,  S = s'c - c's,  n = sqrt(C C + S S),  C /= n,  S /= n,
 *   x' = x C - y S,  y' = y C + x S,  then round to bf16 (nearest even);
 * p' == p copies the stored bits.  V rows are copied.  policy->rope_layout
 * and policy->rotary_dim select the pairs (see KVC_ROPE_*): only the first
 * rotary_dim elements rotate, the rest are copied.
 * PASK App. B.5: a quantised pool stores symmetric codes of the bf16 row:
 * per group a = max|x|, scale = a / qmax rounded to the scale format
 * (nearest even) and raised to its smallest positive value, code =
 * round-half-even(x / scale) clipped to [-qmax, qmax], qmax 7 (int4) or 127
 * (int8); an all-zero group stores zero codes and scale 1.
 *
 * k_cache, v_cache  bf16 [B][L][H_kv][T][d], as for kvc_score.
 * pos_in       int32 [U][T] physical position of each cached row.
 *              These three may also be page-locked host memory registered
 *              with CUDA (cudaHostAlloc, cudaHostRegister): the kept rows
 *              are then read in place through the device mapping, so a cache
 *              offloaded to host memory is not copied whole.  Unregistered
 *              host memory: KVC_ERR_INVALID_ARG.
 * kept_idx, kept_count  as written by kvc_select.
 * rope_cos, rope_sin    fp32 [rope_max_pos][d/2]: cos / sin of p theta_i.
 *              Every old and new position must be < rope_max_pos; a row
 *              whose index or position is out of range is skipped and its
 *              unit marked KVC_UNIT_BAD_INDEX.
 * pools        output arrays (see kvc_pools).
 * unit_status  optional int32 [U]; only errors are written.
 * ---------------------------------------------------------------------- */
kvc_status kvc_compact_rerotate_quant(const kvc_shape* shape, const kvc_policy* policy,
                                      const void* k_cache, const void* v_cache,
                                      const int32_t* pos_in, const int32_t* kept_idx,
                                      const int32_t* kept_count, const float* rope_cos,
                                      const float* rope_sin, int64_t rope_max_pos,
                                      const kvc_pools* pools, int32_t* unit_status,
                                      kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_compact_rerotate_quant_ref -- kvc_compact_rerotate_quant with a
 * reference store for keys (non-compounding re-rotation).
 *
 * PACE Sec. 3.2 and App. D: re-rotating the stored bf16 key at every
 * renumber adds one rounding per position change.  Instead, at a key's
 * first position-changing renumber a copy of its stored bits is kept with
 * the position p_ref it is valid at, and every later position is derived
 * from that copy (same fp32 re-rotation as above, p_ref -> p').  Before use
 * the copy is checked: re-rotated from p_ref to the key's current position
 * p it must reproduce the stored key bit for bit; if it does not, the
 * stored key is re-rotated (p -> p') and becomes the new reference, and the
 * unit's failure counter is incremented.  A key whose position does not
 * change keeps its stored bits and its reference (or none).  References
 * move with the slot: the kept row's reference is written beside it.
 *
 * ref.ref_k        bf16 [U][T][d]: reference copy of every cached key
 *                  (contents ignored where ref_pos < 0); 16-byte aligned.
 * ref.ref_pos      int32 [U][T]: p_ref, or -1 for "no reference".
 * ref.ref_k_out    bf16 [KVC_N_POOLS][U][capacity][d]: references of the
 *                  kept rows (zeros where none); 16-byte aligned.
 * ref.ref_pos_out  int32 [KVC_N_POOLS][U][capacity]: their p_ref (-1: none).
 * ref.failures     optional int32 [U]: incremented once per kept key whose
 *                  reference failed the check (the caller zeroes it).
 * Every other argument and the behaviour of V rows, positions, pools and
 * errors are those of kvc_compact_rerotate_quant.
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* ref_k;
  const int32_t* ref_pos;
  void* ref_k_out;
  int32_t* ref_pos_out;
  int32_t* failures;
} kvc_ref_store;

kvc_status kvc_compact_rerotate_quant_ref(const kvc_shape* shape, const kvc_policy* policy,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* pos_in, const int32_t* kept_idx,
                                          const int32_t* kept_count, const float* rope_cos,
                                          const float* rope_sin, int64_t rope_max_pos,
                                          const kvc_ref_store* ref, const kvc_pools* pools,
                                          int32_t* unit_status, kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_decode_attn -- one decode-attention step over the compacted pools
 * (step a7, the consumer check).
 *
 * PASK Eq. 1 over all kept rows of every pool of the unit, dequantised
 * (x = code * scale); PASK App. B.5: fp32 scores, softmax statistics and
 * accumulation, bf16 output; split partitions are merged by Eq. 15.
 * q    bf16 [B][L][H_q][d], rotated at the decode position.
 * out  bf16 [B][L][H_q][d]; a unit with no kept rows outputs zeros.
 * softmax_scale <= 0 selects 1 / sqrt(d).
 * workspace >= kvc_decode_workspace_bytes(shape, policy), 256-byte aligned.
 * ---------------------------------------------------------------------- */
size_t kvc_decode_workspace_bytes(const kvc_shape* shape, const kvc_policy* policy);
kvc_status kvc_decode_attn(const kvc_shape* shape, const kvc_policy* policy, const void* q,
                           const kvc_pools* pools, const int32_t* kept_count,
                           float softmax_scale, void* out, void* workspace,
                           size_t workspace_bytes, kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_decode_attn_noalloc -- kvc_decode_attn without a caller workspace.
 *
 * Not a step of the pages' methods (they have no counterpart): a variant for
 * callers that cannot allocate device memory -- an engine whose allocator
 * already owns nearly all of HBM, a plug-in that only receives its host
 * framework's buffers, or a latency-critical loop that cannot afford
 * cudaMalloc's implicit synchronisation.  The split-partition scratch lives
 * in a static device array of 2 MiB inside the library, held by every device
 * that loads it until the process exits.  The caller still passes inputs
 * and outputs; the result equals kvc_decode_attn's.
 *   - Returns KVC_ERR_WORKSPACE if kvc_decode_workspace_bytes(shape, policy)
 *     exceeds 2 MiB (nothing is launched).
 *   - Calls no cudaMalloc / cudaFree.  The first call on a device looks up
 *     the array's device address (cudaGetSymbolAddress) and caches it with
 *     the device's current context; make that first call before any stream
 *     capture.  After cudaDeviceReset the device has a new context, and the
 *     next call looks the address up again (again outside any capture).
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; nothing in it needs to start at zero (every partition
 *     slot the merge reads is written earlier in the same call).  Calls that
 *     overlap on the GPU (concurrent streams) race on it: serialise them.
 * ---------------------------------------------------------------------- */
kvc_status kvc_decode_attn_noalloc(const kvc_shape* shape, const kvc_policy* policy,
                                   const void* q, const kvc_pools* pools,
                                   const int32_t* kept_count, float softmax_scale, void* out,
                                   kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_engine_attn -- the engine's attention over persistent, recent and
 * current storage (PASK App. B.5, "Packed attention and quantization").
 *
 * Every visible key appears once across the storages: the persistent pools
 * of a compaction pass (bf16 high map, int8 / int4 low maps dequantised
 * inline as code * scale), the recent storage and the current KV (bf16).  A
 * key at logical position p_k is visible to a query at position p_q iff
 * p_k <= p_q, whatever storage holds it.  For query head h (reading KV head
 * h / G) and query i:
 *   out[h][i] = sum_j softmax_j(q_hi . k_j * scale) v_j over the visible keys,
 * one softmax over all storages (partitions merged by Eq. 15); fp32
 * arithmetic, bf16 output; a query that sees no key outputs 0.  G n_q <= 16
 * (one head, GQA-2, GQA-4, GQA-8; several queries per head for chunked or
 * speculative decoding); rows are split across CTAs (split-KV).
 *
 * q        bf16 [B][L][H_q][n_q][d]; out bf16, same layout.
 * q_pos    optional int32 [B][n_q] (NULL: every key visible).
 * pools    optional (NULL: no persistent storage): the pools of
 *          kvc_compact_rerotate_quant with `policy` (its quant_mode and mode
 *          decide which pools hold rows) and kept_count int32 [KVC_N_POOLS][U];
 *          pools->pos_out gives their positions (required when q_pos is given).
 * recent, current  optional bf16 row stores (NULL or count NULL: empty);
 *          pos NULL = every row visible; k, v 16-byte aligned.
 * workspace >= kvc_engine_attn_workspace_bytes(...), 256-byte aligned (may
 *          be 0 bytes: then NULL is accepted).
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* k;          /* bf16 [U][capacity][d] */
  const void* v;          /* bf16 [U][capacity][d] */
  const int32_t* pos;     /* optional int32 [U][capacity]: logical positions */
  const int32_t* count;   /* int32 [U]: rows in use (<= capacity) */
  int32_t capacity;
} kvc_bf16_rows;

size_t kvc_engine_attn_workspace_bytes(const kvc_shape* shape, const kvc_policy* policy, int32_t n_q,
                                       const kvc_bf16_rows* recent, const kvc_bf16_rows* current);
kvc_status kvc_engine_attn(const kvc_shape* shape, const kvc_policy* policy, const void* q,
                           int32_t n_q, const int32_t* q_pos, const kvc_pools* pools,
                           const int32_t* kept_count, const kvc_bf16_rows* recent,
                           const kvc_bf16_rows* current, float softmax_scale, void* out,
                           void* workspace, size_t workspace_bytes, kvc_stream stream);

/* ------------------------------------------------------------------------
 * CommitKV lifecycle-aware retirement ("CommitKV: Lifecycle-Aware KV Cache
 * Compression via Commit Transitions for Multi-Turn Agents", Sec. 3.2-3.3).
 *
 * An event page is a span [start, start + len) of cache indices, 0 <= len
 * <= 64 (the pages use G = 16); the pages of one call are disjoint.  A
 * window is the last W cache entries (Eq. 5: Q- ends at the tool call's
 * completion, Q+ holds the first W queries of the next turn): row w of query
 * head h sits at index T - W + w and sees indices <= T - W + w, which is
 * "p_i <= p" of Eq. 6 for a cache kept in position order.
 *
 * kvc_deletion_effect -- Eqs. 6-7 for every page and every layer given:
 *   a_rj = softmax_j(q_r . k_j * scale) over the visible keys, o_r = sum a_rj v_j,
 *   s_rE = sum_{j in E} a_rj, u_rE = sum_{j in E} a_rj v_j,
 *   effect[b][l][E] = max over the layer's H_q heads and W rows of
 *       || o_r - (o_r - u_rE) / (1 - s_rE) || / || o_r ||
 *   (+inf if 1 - s_rE <= 0; 0 / +inf if ||o_r|| = 0 and the change is zero /
 *   not zero).  fp32 throughout; the value products use P with 16
 *   significant bits (bf16 head + bf16 tail).
 * k_cache, v_cache  bf16 [B][L][H_kv][T][128]; q_window bf16 [B][L][H_q][W][128]
 *   (rotated); all 16-byte aligned.  head_dim must be 128, W (H_q / H_kv)
 *   <= 64, W <= T.
 * page_start, page_len  int32 [B][n_pages] (the same pages for every layer);
 *   a page outside [0, T) or longer than 64 marks every unit of its sequence
 *   KVC_UNIT_BAD_INDEX in unit_status and counts as empty.
 * effect  fp32 [B][L][n_pages], overwritten.
 * record  caller buffers, all required, overwritten (inputs of
 *   kvc_commit_transition for the post-commit window):
 *     o    fp32 [B][L][H_q][W][128]   window outputs
 *     lse  fp32 [B][L][H_q][W]        natural-log softmax denominators
 *     s    fp32 [B][L][n_pages][H_q][W]
 *     u    fp32 [B][L][n_pages][H_q][W][128]
 * unit_status  optional int32 [U]; KVC_UNIT_TIMEOUT / KVC_UNIT_BAD_INDEX on
 *   failure, untouched otherwise.
 * workspace >= kvc_deletion_effect_workspace_bytes(shape, W), 256-byte
 *   aligned, contents need not be initialised.
 * ---------------------------------------------------------------------- */
typedef struct {
  float* o;
  float* lse;
  float* s;
  float* u;
} kvc_effect_record;

size_t kvc_deletion_effect_workspace_bytes(const kvc_shape* shape, int32_t window);
kvc_status kvc_deletion_effect(const kvc_shape* shape, const void* k_cache, const void* v_cache,
                               const void* q_window, int32_t window, float softmax_scale,
                               const int32_t* page_start, const int32_t* page_len,
                               int32_t n_pages, float* effect, const kvc_effect_record* record,
                               int32_t* unit_status, void* workspace, size_t workspace_bytes,
                               kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_commit_transition -- Eqs. 8-11 on one layer of every sequence.
 *
 * effect_minus, effect_plus  fp32 [B][L][n_pages]: R- and R+ of the same
 *   pages (kvc_deletion_effect over Q- and over Q+); `layer` selects the
 *   attention layer whose effects decide (the page measures one layer).
 * compared  uint8 [B][n_pages]: nonzero = the page is in E_c (both effects
 *   computable).  Percentile rank P(E) = |{E' in E_c : R(E') < R(E)}| / |E_c|.
 * Eq. 9: H = R >= tau_use and P >= rho_use, L = R <= tau_dead and P <= rho_dead.
 * state  uint8 [B][n_pages]: KVC_STATE_* (Eq. 10); KVC_STATE_NOT_COMPARED
 *   outside E_c.
 * retire uint8 [B][n_pages]: 1 = the page joins D_c.  Completion candidates
 *   are tested by increasing R+, then decreasing R-, then lower index; a
 *   candidate joins if R+ of deleting D_c and it together (Eqs. 6-7 on the
 *   combined token set, from record_plus) is <= tau_joint (Eq. 11).
 * joint  optional fp32 [B][n_pages]: the joint R+ each candidate was tested
 *   with; -1 for pages that were not tested.
 * record_plus  the record of the kvc_deletion_effect call over Q+ (same
 *   shape, window and pages).  n_pages <= 1024, H_q W <= 4096.
 * workspace >= kvc_commit_workspace_bytes(shape, W), 256-byte aligned.
 * ---------------------------------------------------------------------- */
enum {
  KVC_STATE_UNCERTAIN = 0,
  KVC_STATE_COMPLETION_CANDIDATE = 1,
  KVC_STATE_DORMANT = 2,
  KVC_STATE_NEWLY_ACTIVE = 3,
  KVC_STATE_STILL_ACTIVE = 4,
  KVC_STATE_NOT_COMPARED = 255
};

typedef struct {
  float tau_use;    /* 0.05 (CommitKV Sec. 4.1) */
  float tau_dead;   /* 0.01 */
  float rho_use;    /* 0.75 */
  float rho_dead;   /* 0.25 */
  float tau_joint;  /* 0.01 */
} kvc_commit_thresholds;

size_t kvc_commit_workspace_bytes(const kvc_shape* shape, int32_t window);
kvc_status kvc_commit_transition(const kvc_shape* shape, int32_t window, int32_t layer,
                                 int32_t n_pages, const float* effect_minus,
                                 const float* effect_plus, const uint8_t* compared,
                                 const kvc_commit_thresholds* thresholds,
                                 const kvc_effect_record* record_plus, uint8_t* state,
                                 uint8_t* retire, float* joint, void* workspace,
                                 size_t workspace_bytes, kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_protect_pending -- Eq. 12: pages awaiting their post-commit
 * measurement (pending != 0) are protected by decreasing R- of layer
 * `layer` (ties: lower index) while the protected token count stays
 * <= budget_tokens (B_N = floor(eta B)) and the page count <= max_pages
 * (the page uses 16); the walk stops at the first page that does not fit.
 * effect_minus fp32 [B][L][n_pages]; pending uint8 [B][n_pages];
 * page_len int32 [B][n_pages]; protect uint8 [B][n_pages] (0 / 1).
 * n_pages <= 1024.
 * ---------------------------------------------------------------------- */
kvc_status kvc_protect_pending(const kvc_shape* shape, int32_t layer, int32_t n_pages,
                               const float* effect_minus, const uint8_t* pending,
                               const int32_t* page_len, int32_t budget_tokens, int32_t max_pages,
                               uint8_t* protect, kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_commit_flags -- the checkpoint's selection flags (Alg. 1, Eq. 13):
 * tokens of protected pages become KVC_FLAG_PROTECT (EXCLUDE cleared), tokens
 * of retired pages that are not protected become KVC_FLAG_EXCLUDE (PROTECT
 * cleared); every other token keeps its flags.  flags uint8 [B][n_tokens]
 * (kvc_policy.flags of token mode), updated in place; retire / protect
 * optional uint8 [B][n_pages]; pages as in kvc_deletion_effect.
 * ---------------------------------------------------------------------- */
kvc_status kvc_commit_flags(int32_t batch, int64_t n_tokens, int32_t n_pages,
                            const int32_t* page_start, const int32_t* page_len,
                            const uint8_t* retire, const uint8_t* protect, uint8_t* flags,
                            kvc_stream stream);

/* ------------------------------------------------------------------------
 * kvc_set_overrides -- process-wide overrides of the launch plans, for
 * tuning sweeps and for failure-detection tests.  Not a step of the pages'
 * methods; a production caller never needs it.  0 in a field keeps the
 * library's own choice:
 *   score_chunk_tiles   key tiles (of 128 rows) per kvc_score work item
 *   decode_splits       split partitions per unit of kvc_decode_attn (<= 32)
 *   effect_chunk_tiles  key tiles per kvc_deletion_effect work item
 *   score_stall_unit    -1 = off.  Test hook: in kvc_score the pass-1 wait
 *                       of this unit never completes, so after the bounded
 *                       wait (2 s) that unit and every unit its CTA leaves
 *                       unscored report KVC_UNIT_TIMEOUT.
 *   select_stall_unit   -1 = off.  Test hook: in kvc_select (token and page
 *                       mode, units of at most 32,768 items whose scores
 *                       are copied to shared memory in bulk) this unit waits
 *                       for 16 bytes more than its copy brings, so after
 *                       the bounded wait (2 s, then 2 s more for the copy)
 *                       it reports KVC_UNIT_TIMEOUT and keeps nothing.
 * NULL restores every default.  Values out of range return
 * KVC_ERR_INVALID_ARG and change nothing.  A call affects calls issued
 * after it from any host thread; it does not synchronise with them.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t score_chunk_tiles;
  int32_t decode_splits;
  int32_t effect_chunk_tiles;
  int32_t score_stall_unit;
  int32_t select_stall_unit;
} kvc_overrides;
kvc_status kvc_set_overrides(const kvc_overrides* overrides);

/* Static text for a status code. */
const char* kvc_status_string(kvc_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
