/*
 * cpattn.h -- C ABI of the GB300 (sm_103a) prefill context-parallel causal
 * attention library.
 *
 * The hot path: shard a batch's new (uncached) query tokens over C logical
 * context-parallel (CP) ranks, compute every shard's causal attention against
 * the gathered KV (one KV buffer in HBM that all shards read) as a partial
 * output O with its log-sum-exp L, merge partials with the log-sum-exp rule
 * and put the result back in causal token order.
 *
 * Sources (the behaviour each call implements is defined there):
 *   [SGL-ZZ]  SGLang docs, "Prefill Context Parallelism", section "Zigzag strategy"
 *   [SGL-IL]  same page, section "Interleave strategy"
 *   [SGL-BE]  same page, section "Attention backend integration"
 *   [CPB-2.1] blog "什么是 Context Parallelism" (zhifeiding), section 2.1
 *             (all-gather KV; restore index after the all-gather)
 *   [CPB-3.3] same blog, sections 3.1 and 3.3 (per-shard partial O_j and LSE L_j)
 *   [CPB-3.6] same blog, section 3.6 (merging partials: online-softmax / LSE rule)
 *   [CPB-3.5] same blog, section 3.5, the pass-KV / pass-Q switch (miss-rate
 *             rule and fitted heuristic)
 *   [CPB-PQ]  same blog, section 3.3.2 "Pass Q" (ring pass-Q: the query block
 *             carries a partial accumulator (O_acc, L_acc) from rank to rank
 *             and every hop merges its local partial into it)
 *
 * Conventions for every call:
 *   - Return value: CPATTN_OK (0) or a negative CPATTN_ERR_* code.  Argument
 *     errors are detected on the host and returned synchronously; nothing is
 *     launched then.  No C++ exception crosses this boundary.
 *   - Device work is asynchronous on the given stream.  Errors detected on the
 *     device (bad segment metadata, an index out of range, a pipeline wait that
 *     ran out) are written to the optional device word *status_dev (first error
 *     wins; the caller zeroes it) and the offending work is skipped; the kernel
 *     never traps.
 *   - Ownership: the caller allocates and owns every buffer.  The library
 *     allocates no device or host memory and writes only to output pointers.
 *   - Device pointers must be 16-byte aligned unless a call states otherwise
 *     (checked: CPATTN_ERR_ALIGNMENT).
 *   - Tokens: the batch's new tokens are flattened in request order ("flat
 *     index").  Request b has new_lens[b] new tokens at positions
 *     prefix_lens[b] .. prefix_lens[b]+new_lens[b]-1 (positions count the
 *     cached prefix).  The KV buffer holds, per request in batch order, key
 *     positions 0 .. prefix_lens[b]+new_lens[b]-1 (prefix first).
 *   - Shard order: "cat" rows are all shards' rows concatenated in rank order
 *     (rank 0's rows, then rank 1's, ...): the layout an all-gather produces.
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPATTN_OK 0
#define CPATTN_ERR_INVALID_ARG (-1)  /* bad size, count, enum or metadata */
#define CPATTN_ERR_UNSUPPORTED (-2)  /* valid but unsupported shape (head dims, ...) */
#define CPATTN_ERR_CUDA (-3)         /* a CUDA runtime/driver call failed */
#define CPATTN_ERR_TIMEOUT (-4)      /* device: a pipeline wait exceeded its time limit */
#define CPATTN_ERR_ALIGNMENT (-5)    /* a pointer or stride is not 16-byte aligned */
#define CPATTN_ERR_RANGE (-6)        /* device: an index or segment lies outside its buffer */
#define CPATTN_ERR_TOO_LARGE (-7)    /* the problem needs more scratch than the static buffer */

typedef enum { CP_ZIGZAG = 0, CP_INTERLEAVE = 1 } cp_strategy_t;

/* One segment: a maximal run of one rank's query rows that belong to one
 * request and whose positions advance by a constant step.  Row i of the
 * segment (0 <= i < q_len) is cat row q_row0 + i, has position
 * q_pos0 + i * q_pos_step and flat index tok0 + i * q_pos_step, and attends to
 * key positions 0 .. its position (KV rows kv_row0 + key position).
 * Zigzag: one segment per non-empty block, q_pos_step = 1.  Interleave: one
 * segment per (rank, request) with rows in it, q_pos_step = C.
 * [SGL-ZZ] "separate query and KV lengths for the early and late blocks,
 * including any cached prefix"; [SGL-IL] "per-request sharding metadata
 * preserves those boundaries and each query's causal extent". */
typedef struct {
  int32_t q_row0;     /* first cat row of the segment */
  int32_t q_len;      /* rows in the segment (> 0) */
  int32_t q_pos0;     /* position of row 0 within its request (prefix counted) */
  int32_t q_pos_step; /* position (and flat index) increment per row; plans
                         produce >= 1, attention also accepts 0 (all rows at
                         one position, e.g. decode-style queries) */
  int32_t kv_row0;    /* KV-buffer row of the request's key position 0 */
  int32_t kv_len;     /* keys visible to the segment's last row = its position + 1 */
  int32_t tok0;       /* flat index of row 0 */
  int32_t req;        /* request index */
} cp_segment_t;

/* Query tiles of the attention kernel are this many rows of one segment. */
#define CPATTN_TILE_ROWS 128

/* ------------------------------------------------------------------------ */
/* Plan sizes (host only, no device work).  [SGL-ZZ], [SGL-IL]
 *   new_lens, prefix_lens: host arrays [num_reqs], entries >= 0.
 *   num_reqs in [0, CPATTN_MAX_REQS]; cp_size in [1, CPATTN_MAX_CP].
 * Outputs (host arrays [cp_size], any may be NULL): rows, segments and
 * CPATTN_TILE_ROWS-row tiles owned by each rank.  The plan buffers of
 * cp_shard_plan are sized from their sums.  Totals must stay below 2^31. */
#define CPATTN_MAX_REQS 65536
#define CPATTN_MAX_CP 1024
int cp_shard_plan_sizes(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                        int cp_size, int strategy, int32_t* rows_per_rank,
                        int32_t* segs_per_rank, int32_t* tiles_per_rank);

/* Build the shard plan on the device.  [SGL-ZZ], [SGL-IL], [CPB-2.1]
 *   new_lens_dev, prefix_lens_dev: device int32 [num_reqs].
 *   total_rows / total_segs / total_tiles: the sums reported by
 *     cp_shard_plan_sizes for the same lengths (checked on the device;
 *     a mismatch sets CPATTN_ERR_INVALID_ARG in *status_dev).
 * Outputs (device, caller-allocated):
 *   segs_dev        [total_segs]   segments, rank by rank; within a rank in
 *                                  cat-row order.  Zigzag: request by request,
 *                                  early block (r) before late block (2C-1-r).
 *   seg_offsets_dev [cp_size+1]    first segment of each rank
 *   row_offsets_dev [cp_size+1]    first cat row of each rank
 *   gather_idx_dev  [total_rows]   cat row -> flat index
 *   positions_dev   [total_rows]   cat row -> position within its request
 *   restore_idx_dev [total_rows]   flat index -> cat row (the restore index)
 *   tiles_dev       [total_tiles]  (nullable) CPATTN_TILE_ROWS-row query tiles
 *                                  as int32 pairs (segment, tile-in-segment),
 *                                  heaviest first (descending count of keys
 *                                  visible to the tile's last row); the order
 *                                  among equal counts is unspecified.
 *   status_dev      (nullable)     device error word. */
int cp_shard_plan(const int32_t* new_lens_dev, const int32_t* prefix_lens_dev, int num_reqs,
                  int cp_size, int strategy, int total_rows, int total_segs, int total_tiles,
                  cp_segment_t* segs_dev, int32_t* seg_offsets_dev, int32_t* row_offsets_dev,
                  int32_t* gather_idx_dev, int32_t* positions_dev, int32_t* restore_idx_dev,
                  int32_t* tiles_dev, int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Causal attention of shard rows against the gathered KV, giving the partial
 * output O and its log-sum-exp L.  [SGL-BE], [CPB-3.3]
 *
 * For every row of every segment and every query head h, with
 * P = the row's position and key window [lo, hi) = [max(kv_lo,0), min(kv_hi, P+1))
 * (kv_hi < 0 means unbounded):
 *     S_k = scale * q[h] . K[kv_row0 + k, h / (Hq/Hkv)]      for k in [lo, hi)
 *     L   = ln(sum_k exp(S_k))
 *     O   = sum_k exp(S_k - L) * V[kv_row0 + k, h / (Hq/Hkv)]
 * An empty window gives O = 0 and L = -inf (the identity of cp_lse_merge).
 *
 *   segs_dev, num_segs: segments (e.g. from cp_shard_plan, or a sub-range).
 *   tiles_dev, num_tiles: (nullable) tile list from cp_shard_plan restricted to
 *     these segments, in launch order (heaviest first).  NULL: all tiles of
 *     all segments in segment order.
 *   q:  bf16 [num_q_rows, Hq, d] (cat rows), contiguous.
 *   k:  bf16 key rows; element (row, head, c) at k[row*k_row_stride + head*k_head_stride + c].
 *   v:  bf16 value rows, same with v_row_stride / v_head_stride (v may alias k:
 *       absorbed MLA passes v = k with the latent as the first dv columns).
 *   num_kv_rows: rows addressable through k and v.
 *   Hq % Hkv == 0.  Supported (d, dv): (64, 64), (128, 128) and the absorbed-MLA
 *   shape (576, 512), which requires v == k with equal strides (the value is
 *   the first 512 columns of each key row); other shapes: CPATTN_ERR_UNSUPPORTED.
 *   o:  [num_out_rows, Hq, dv], bf16 (o_is_fp32 = 0) or fp32 (o_is_fp32 = 1);
 *       segment row with cat row R is written at output row R - out_row_base.
 *   lse: fp32 [num_out_rows, Hq] (natural log), same row mapping.
 * Every row of every segment (and tile) is written exactly once.  Segments
 * that point outside q, k, v or o set CPATTN_ERR_RANGE and are skipped. */
int cp_attn_partial(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev,
                    int num_tiles, const void* q, int num_q_rows, const void* k,
                    int64_t k_row_stride, int64_t k_head_stride, const void* v,
                    int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq,
                    int Hkv, int d, int dv, float scale, int kv_lo, int kv_hi, void* o,
                    int o_is_fp32, float* lse, int out_row_base, int num_out_rows,
                    int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Full-KV CP attention in original token order.  [SGL-ZZ], [SGL-BE],
 * [CPB-2.1]
 *
 * cp_attn_partial over the whole key range, with every segment row addressed
 * by its token (flat) index: segment row i reads query row tok0 + i of q and
 * writes output row tok0 + i of o and lse.  The shard gather of the queries
 * and the restore of the outputs are thus done by the kernel's own loads and
 * stores.  Every segment must be a run of consecutive tokens (q_pos_step == 1:
 * the segments of a zigzag plan, or of any plan with cp_size 1); another one
 * sets CPATTN_ERR_RANGE and is skipped.
 *   q: bf16 [num_tokens, Hq, d] in original order; o: [num_tokens, Hq, dv]
 *   bf16 or fp32; lse: fp32 [num_tokens, Hq].  Other arguments as in
 *   cp_attn_partial. */
int cp_attn_prefill(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev,
                    int num_tiles, const void* q, int num_tokens, const void* k,
                    int64_t k_row_stride, int64_t k_head_stride, const void* v,
                    int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq,
                    int Hkv, int d, int dv, float scale, void* o, int o_is_fp32, float* lse,
                    int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* cp_attn_partial with the restore fused into the store.  [CPB-2.1] (the
 * restore index after the all-gather), [SGL-BE]
 *
 * Same computation and arguments as cp_attn_partial, except that the output
 * row of query (cat) row i is dst_rows[i] instead of i - out_row_base.  With
 * dst_rows = the plan's gather index (cat row -> flat index) the shard outputs
 * land directly in causal token order, so no cp_restore pass is needed.
 *   dst_rows: device int32 [num_q_rows]; every entry used must lie in
 *     [0, num_out_rows) (an entry outside sets CPATTN_ERR_RANGE and that row
 *     is not written).  Rows are written once each if dst_rows is injective on
 *     the segments' rows; otherwise the last writer wins (unspecified).
 *   o: [num_out_rows, Hq, dv] bf16 or fp32; lse: fp32 [num_out_rows, Hq]. */
int cp_attn_partial_restore(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev,
                            int num_tiles, const void* q, int num_q_rows, const void* k,
                            int64_t k_row_stride, int64_t k_head_stride, const void* v,
                            int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq,
                            int Hkv, int d, int dv, float scale, int kv_lo, int kv_hi,
                            const int32_t* dst_rows, void* o, int o_is_fp32, float* lse,
                            int num_out_rows, int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* One pass-Q hop: cp_attn_partial whose store merges the new partial into a
 * running accumulator.  [CPB-PQ], [CPB-3.6]
 *
 * For every segment row (output row R = cat row - out_row_base) and head h,
 * with (O_new, L_new) = cp_attn_partial's result for the key window
 * [kv_lo, kv_hi) and (O_acc, L_acc) = o_acc[R, h, :], lse_acc[R, h]:
 *     m = max(L_acc, L_new);  w_a = exp(L_acc - m);  w_n = exp(L_new - m)
 *     o_acc[R, h, :]  <- (w_a O_acc + w_n O_new) / (w_a + w_n)
 *     lse_out[R, h]   <- m + ln(w_a + w_n)
 * and both empty (L = -inf) gives O = 0, L = -inf.  An accumulator that starts
 * at O = 0, L = -inf (the identity) and goes through hops whose windows
 * partition the keys ends equal to cp_attn_partial over all keys.
 *   Arguments shared with cp_attn_partial keep its meaning.
 *   seg_windows_dev: nullable int32 [num_segs][2] on the device, 4-byte
 *     aligned.  When set, segment s uses its own key window
 *     [seg_windows_dev[2s], seg_windows_dev[2s+1]) (upper end < 0:
 *     unbounded) and kv_lo / kv_hi are ignored, so that one launch can
 *     merge every visiting shard against its own rank's resident KV block
 *     (one launch per ring hop and block instead of one per rank).
 *   o_acc: fp32 [num_out_rows, Hq, dv], read and overwritten in place.
 *   lse_acc: fp32 [num_out_rows, Hq] read; lse_out: fp32 [num_out_rows, Hq]
 *     written.  The two must not overlap (CPATTN_ERR_INVALID_ARG): a hop
 *     reads the old LSE of a row from more than one thread block (the MLA
 *     shape splits dv over two), so the caller alternates two LSE buffers.
 *   Rows outside the segments are not touched. */
int cp_attn_partial_accumulate(const cp_segment_t* segs_dev, int num_segs,
                               const int32_t* tiles_dev, int num_tiles, const void* q,
                               int num_q_rows, const void* k, int64_t k_row_stride,
                               int64_t k_head_stride, const void* v, int64_t v_row_stride,
                               int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv, int d,
                               int dv, float scale, int kv_lo, int kv_hi,
                               const int32_t* seg_windows_dev, float* o_acc,
                               const float* lse_acc, float* lse_out, int out_row_base,
                               int num_out_rows, int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Pass-KV or pass-Q for one step.  [CPB-3.5]  Host only; no device work.
 *
 * new_tokens T > 0 (uncached tokens of the step), cached_tokens P >= 0
 * (persistent KV length), both at most 2^40; Hq / Hkv query / KV heads
 * (Hq % Hkv == 0, Hq <= 2^20).
 *   rule CP_SELECT_MESSAGE: pass-Q iff the miss rate T/(T+P) <= 2*Hkv/Hq,
 *     i.e. iff the query block (T x Hq heads) is no larger than the K and V
 *     block (T+P rows x Hkv heads each) that pass-KV would send (decided
 *     exactly in integers: T*Hq <= 2*(T+P)*Hkv); *score =
 *     T/(T+P) - 2*Hkv/Hq (> 0: pass-KV).
 *   rule CP_SELECT_FITTED: the blog's fitted heuristic
 *     h(T,P) = -1.059 log T + 1.145 log(T/(T+P)) + 12.112, pass-KV iff h > 0,
 *     read with natural logarithms of token counts (the page gives no base
 *     or unit); *score = h.
 *   score: nullable.
 * Returns CP_PASS_KV or CP_PASS_Q, or CPATTN_ERR_INVALID_ARG. */
#define CP_PASS_KV 0
#define CP_PASS_Q 1
#define CP_SELECT_MESSAGE 0
#define CP_SELECT_FITTED 1
int cp_select_pass(int64_t new_tokens, int64_t cached_tokens, int Hq, int Hkv, int rule,
                   double* score);

/* Pass-KV or pass-Q by cost, from measured rates.  [CPB-3.5]  Host only.
 * The page lays a roofline condition over the message comparison (pass-KV is
 * preferred when its per-hop SendRecv hides behind that hop's attention) and
 * refines pass-Q with the All2All that returns its scattered partials before
 * the LSE merge.  This call prices both for one rank of a ring of cp_size
 * ranks (T = new_tokens, P = cached_tokens, d = head_dim = dv, bf16 messages,
 * fp32 partials):
 *   F     = 2 Hq 2d (T P + T (T+1) / 2)          attention flops of the step
 *   t_a   = F / C^2 / (attn_tflops 1e12)         attention of one hop
 *   t_kv  = 2 ceil((T+P)/C) Hkv d 2 / (link_gbs 1e9)      K and V of one hop
 *   t_q   = ceil(T/C) Hq d 2 / (link_gbs 1e9)             Q of one hop
 *   t_a2a = (C-1)/C ceil(T/C) Hq (d+1) 4 / (link_gbs 1e9) the All2All
 *   t_m   = C ceil(T/C) Hq (d+1) 4 / (merge_gbs 1e9)      the final merge
 *   E_kv  = (C-1) max(0, t_kv - t_a)
 *   E_q   = (C-1) max(0, t_q - t_a) + t_a2a + t_m
 * and returns CP_PASS_KV iff E_kv <= E_q, else CP_PASS_Q.  attn_tflops and
 * merge_gbs are meant to be this library's measured attention and merge
 * rates; link_gbs the per-GPU ring bandwidth.  exposed_kv_s / exposed_q_s
 * (nullable) receive E_kv and E_q in seconds.  Arguments as cp_select_pass,
 * plus head_dim in [1, 4096], cp_size in [1, CPATTN_MAX_CP] and positive
 * finite rates; otherwise CPATTN_ERR_INVALID_ARG. */
int cp_select_pass_cost(int64_t new_tokens, int64_t cached_tokens, int Hq, int Hkv, int head_dim,
                        int cp_size, double attn_tflops, double link_gbs, double merge_gbs,
                        double* exposed_kv_s, double* exposed_q_s);

/* ------------------------------------------------------------------------ */
/* Partial-KV (ring-style) decomposition in one call.  [CPB-2.1] item 2,
 * [CPB-3.3] (pass-KV: a rank's queries meet the KV one block at a time, each
 * block giving (O_j, L_j)), [CPB-3.6] (the merge).
 *
 * Every segment's keys are cut into blocks of kv_block key positions, block j
 * = [j*kv_block, (j+1)*kv_block); a segment whose last row is at position P
 * sees blocks 0 .. P / kv_block.  For every visible (segment, block) pair and
 * every head, the fp32 partial (O_j, L_j) of cp_attn_partial with that window
 * is written to the workspace (one launch over all pairs), then the partials
 * of each row are LSE-merged (cp_lse_merge's rule) and written to output row
 * dst_rows[cat row] (dst_rows non-NULL: e.g. the plan's gather index, which
 * restores causal order) or to the cat row.  The result equals cp_attn_partial
 * over the full window up to rounding.
 *
 *   Arguments shared with cp_attn_partial keep its meaning.
 *   kv_block > 0; max_blocks: an upper bound on the blocks any segment sees,
 *     1 <= max_blocks <= 32 (a segment with more sets CPATTN_ERR_INVALID_ARG).
 *   max_seg_rows: an upper bound on every segment's q_len, or 0 when unknown.
 *     With 1 <= max_seg_rows <= CPATTN_TILE_ROWS / 2 (a decode step's few
 *     queries) and Hq / Hkv a multiple of 4 (d = 64 or 128), each 128-row
 *     query tile holds two query heads of the same KV head.  That halves the
 *     tiles and the MMA work of short segments.  A segment longer than a
 *     bound that enabled packing sets CPATTN_ERR_RANGE and is skipped.
 *     With num_segs == 0 the call does nothing and returns CPATTN_OK, and
 *     max_blocks may be 0 (what the sizing calls report for a batch without
 *     new tokens).
 *   dst_rows: nullable, [num_q_rows] output row of each cat row.
 *   o_out: [num_out_rows, Hq, dv] bf16 or fp32; lse_out fp32 [num_out_rows, Hq]
 *     (nullable).
 *   workspace: device scratch of workspace_bytes (16-byte aligned), at least
 *     cp_partial_kv_workspace_size for the plan's lengths; its contents are
 *     overwritten.  Too small: CPATTN_ERR_INVALID_ARG in *status_dev and the
 *     partials that do not fit are skipped.
 * Three launches on the stream (layout, attention, merge); the attention and
 * the merge use programmatic dependent launch, so each may start while the
 * launch before it in the call is still running (the layout kernel itself
 * waits for earlier work on the stream like any launch). */
/* Sizing (host only).  bytes: the workspace for the segments cp_shard_plan
 * makes from these lengths; max_blocks (nullable): the largest block count of
 * any segment, the value to pass to cp_attn_partial_kv; max_seg_rows
 * (nullable): the longest segment's q_len, the value to pass as
 * max_seg_rows (it turns on head packing when it is at most
 * CPATTN_TILE_ROWS / 2). */
int cp_partial_kv_workspace_size(const int32_t* new_lens, const int32_t* prefix_lens,
                                 int num_reqs, int cp_size, int strategy, int kv_block, int Hq,
                                 int dv, int64_t* bytes, int32_t* max_blocks,
                                 int32_t* max_seg_rows);
/* The same sizing for an explicit segment table on the host (for segments
 * that no plan made, e.g. a decode step's few queries over a KV shard):
 * bytes, the largest block count and the longest segment over
 * segs_host[0 .. num_segs). */
int cp_partial_kv_workspace_size_segs(const cp_segment_t* segs_host, int num_segs, int kv_block,
                                      int Hq, int dv, int64_t* bytes, int32_t* max_blocks,
                                      int32_t* max_seg_rows);
int cp_attn_partial_kv(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev,
                       int num_tiles, const void* q, int num_q_rows, const void* k,
                       int64_t k_row_stride, int64_t k_head_stride, const void* v,
                       int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq,
                       int Hkv, int d, int dv, float scale, int kv_block, int max_blocks,
                       int max_seg_rows, const int32_t* dst_rows, void* o_out, int o_is_fp32,
                       float* lse_out,
                       int num_out_rows, void* workspace, int64_t workspace_bytes,
                       int32_t* status_dev, cudaStream_t stream);

/* The same computation as cp_attn_partial_kv, for callers that cannot
 * allocate device memory: a framework or serving engine whose allocator owns
 * all device memory, a deployment with a fixed memory budget set at start-up,
 * or a hot path that cannot take the implicit synchronisation of cudaMalloc /
 * cudaFree.  There is no counterpart on the source pages.
 *   The caller still passes inputs and outputs; the scratch is a static device
 *   array of CPATTN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU
 *   that loads the library keeps until the process exits.
 *   workspace_bytes_needed: what cp_partial_kv_workspace_size reports for
 *     the plan's lengths.  Above CPATTN_NOALLOC_SCRATCH_BYTES the call returns
 *     CPATTN_ERR_TOO_LARGE and launches nothing.  This host check trusts the
 *     caller's figure: if the figure is too small and the real need exceeds
 *     the array, the call launches and the device reports it as
 *     cp_attn_partial_kv does for a small workspace (CPATTN_ERR_INVALID_ARG in
 *     *status_dev, the partials that do not fit skipped); nothing is written
 *     past the array.
 *   The first call in a CUDA context looks up the scratch address in that
 *   context (cudaGetSymbolAddress, with the device current) and caches it
 *   under the context's unique id; make that first call before any stream
 *   capture.  A new context on the device (e.g. after cudaDeviceReset) has a
 *   new id, so its first call looks the address up again, also outside any
 *   capture.  The call allocates nothing (no cudaMalloc/cudaFree).
 *   All calls share one scratch array, which keeps the last call's contents:
 *   calls that overlap on the GPU (other streams, other host threads) race on
 *   it and must be serialised by the caller.  Nothing in it needs clearing.
 * Other arguments and errors: as cp_attn_partial_kv. */
#define CPATTN_NOALLOC_SCRATCH_BYTES (64 << 20)
int cp_attn_partial_kv_noalloc(const cp_segment_t* segs_dev, int num_segs,
                               const int32_t* tiles_dev, int num_tiles, const void* q,
                               int num_q_rows, const void* k, int64_t k_row_stride,
                               int64_t k_head_stride, const void* v, int64_t v_row_stride,
                               int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv, int d,
                               int dv, float scale, int kv_block, int max_blocks,
                               int max_seg_rows, const int32_t* dst_rows, void* o_out,
                               int o_is_fp32,
                               float* lse_out, int num_out_rows, int64_t workspace_bytes_needed,
                               int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Pass-Q ring: schedule (host only) and the whole ring in one call.
 * [CPB-PQ]; [CPB-3.5] (the persistent KV cache split into 2C first/last-paired
 * blocks).
 *
 * KV residency: each request's key positions 0 .. p+n-1 are cut into 2C blocks
 * like the zigzag query split (block k has (p+n)/2C keys plus one when
 * k < (p+n) mod 2C) and rank r keeps blocks r and 2C-1-r.  At ring hop s
 * (0 <= s < C) the query shard of rank q is on rank (q+s) mod C.  Launch
 * (s, b), b in {0, 1}, holds every segment of the plan (cp_shard_plan's
 * table order) whose request's resident block b on its host rank is non-empty
 * and starts at or before the segment's last position, with that block as the
 * segment's key window.  Launches run hop-major, block-minor; empty ones are
 * left out, so num_launches <= 2C.
 *
 * cp_pass_q_schedule_size: num_launches and num_entries (total segment
 *   entries over all launches), to size the buffers below.
 * cp_pass_q_schedule (host arrays, caller-allocated):
 *   launch_first [num_launches+1]  first entry of each launch, then num_entries
 *   launch_hop, launch_block [num_launches]  (nullable) s and b of each launch
 *   entry_segs [num_entries]       copies of the plan's segment rows
 *   entry_windows [2*num_entries]  key window [lo, hi) of each entry
 *   entry_seg_ids [num_entries]    (nullable) index of the entry's segment in
 *                                  the plan's segment table
 * Arguments as cp_shard_plan_sizes; errors CPATTN_ERR_INVALID_ARG. */
int cp_pass_q_schedule_size(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                            int cp_size, int strategy, int32_t* num_launches,
                            int32_t* num_entries);
int cp_pass_q_schedule(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                       int cp_size, int strategy, int32_t* launch_first, int32_t* launch_hop,
                       int32_t* launch_block, cp_segment_t* entry_segs, int32_t* entry_windows,
                       int32_t* entry_seg_ids);

/* The pass-Q ring on the device: the accumulator starts at the identity
 * (O = 0, L = -inf) and every launch of the schedule merges its entries'
 * partials into it (cp_attn_partial_accumulate with per-segment windows).
 * After the last launch every row holds attention over all its visible keys.
 *   entry_segs_dev, entry_windows_dev: the schedule's entry arrays copied to
 *     the device (16- and 4-byte aligned).  launch_first: HOST int32
 *     [num_launches+1] from cp_pass_q_schedule.
 *   q, k, v and shapes: as cp_attn_partial (q in cat order, num_q_rows rows).
 *   o_acc: fp32 [num_q_rows, Hq, dv]; lse: fp32 [num_q_rows, Hq] (natural log);
 *     both written (cat order).  lse_scratch: fp32 [num_q_rows, Hq], scratch
 *     that must not overlap lse.
 * Launches on the stream: one initialisation kernel, then per launch one
 * attention launch and one device-to-device copy of the LSE. */
int cp_attn_pass_q(const cp_segment_t* entry_segs_dev, const int32_t* entry_windows_dev,
                   const int32_t* launch_first, int num_launches, const void* q, int num_q_rows,
                   const void* k, int64_t k_row_stride, int64_t k_head_stride, const void* v,
                   int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv,
                   int d, int dv, float scale, float* o_acc, float* lse, float* lse_scratch,
                   int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Host-to-host full-KV CP prefill of a sequence of same-shaped batches (the
 * end-to-end path).  [SGL-ZZ], [SGL-IL], [SGL-BE], [CPB-2.1]
 *
 * Batch i (0 <= i < num_batches) has host inputs q_host[i] bf16 [N, Hq, d] in
 * original token order, k_host[i] bf16 [KV, Hkv, d] and v_host[i] bf16
 * [KV, Hkv, dv] (KV rows as in cp_attn_partial; with v_is_k_prefix the value
 * is the first dv columns of each key row, v_host is ignored and may be NULL,
 * as for the absorbed MLA shape), and host outputs o_host[i] bf16 [N, Hq, dv]
 * and lse_host[i] fp32 [N, Hq], in original token order.  N and KV follow
 * from new_lens / prefix_lens (host arrays [num_reqs]).
 * Per batch: its inputs are copied in on `upload`; on `compute` the plan is
 * built (cp_shard_plan) and every shard attends to the gathered KV (zigzag:
 * cp_attn_prefill; interleave: cp_restore of the queries into shard order and
 * cp_attn_partial_restore); O and LSE are copied out on `download`.  Two
 * device buffer sets let batch i's attention overlap batch i+1's upload and
 * batch i-1's download.  The streams may be the same stream (then nothing
 * overlaps).  The call returns once everything is queued; the outputs are
 * valid once `download` has completed.  Host buffers should be page-locked
 * for the copies to run asynchronously, and must stay valid until then.
 *   workspace: device memory of at least cp_prefill_host_workspace_size bytes,
 *     256-byte aligned, owned by the caller (plan buffers and two buffer sets).
 *   The call creates and destroys six CUDA events (no memory is allocated).
 * Errors: argument errors as CPATTN_ERR_* before anything is queued; a failed
 * CUDA call returns CPATTN_ERR_CUDA (work queued before it stays queued);
 * device-detected errors go to *status_dev. */
int cp_prefill_host_workspace_size(const int32_t* new_lens, const int32_t* prefix_lens,
                                   int num_reqs, int cp_size, int strategy, int Hq, int Hkv,
                                   int d, int dv, int v_is_k_prefix, int64_t* bytes);
int cp_prefill_host(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                    int cp_size, int strategy, int Hq, int Hkv, int d, int dv, float scale,
                    int v_is_k_prefix, int num_batches, const void* const* q_host,
                    const void* const* k_host, const void* const* v_host, void* const* o_host,
                    float* const* lse_host, void* workspace, int64_t workspace_bytes,
                    int32_t* status_dev, cudaStream_t compute, cudaStream_t upload,
                    cudaStream_t download);

/* ------------------------------------------------------------------------ */
/* Merge num_parts partial results with the log-sum-exp rule.  [CPB-3.6]
 * For each row i < rows and head h < Hq, partial j has
 *     O_j = o_parts[j*o_part_stride + (i*Hq + h)*dv .. +dv]   (fp32)
 *     L_j = lse_parts[j*lse_part_stride + i*Hq + h]            (fp32, natural log)
 * and the result is
 *     m = max_j L_j,  w_j = exp(L_j - m),  L = m + ln(sum_j w_j),
 *     O = sum_j w_j O_j / sum_j w_j
 * (parts with L_j = -inf have weight 0; all empty gives O = 0, L = -inf).
 * The merged row i is written to output row dst_rows[i] (dst_rows non-NULL:
 * a fused scatter such as the restore to causal order, each entry in
 * [0, num_out_rows)) or row i (dst_rows NULL).  o_out: [num_out_rows, Hq, dv]
 * bf16 or fp32; lse_out: fp32 [num_out_rows, Hq] (nullable).
 * 1 <= num_parts <= 32; dv % 4 == 0 and dv <= 1024. */
int cp_lse_merge(const float* o_parts, const float* lse_parts, int num_parts,
                 int64_t o_part_stride, int64_t lse_part_stride, int rows, int Hq, int dv,
                 const int32_t* dst_rows, void* o_out, int o_out_is_fp32, float* lse_out,
                 int num_out_rows, int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Row gather: dst[i] = src[idx[i]] for i < rows, rows of row_bytes bytes
 * (row_bytes % 4 == 0; src and dst 4-byte aligned; 16-byte rows and
 * pointers take the vectorised path).  With idx = the plan's restore index and src = the
 * all-gathered cat rows this restores causal token order [CPB-2.1]; with idx
 * = the gather index it builds the shard-local (cat) layout from original
 * order.  An index outside [0, num_src_rows) sets CPATTN_ERR_RANGE and its row
 * is left unwritten. */
int cp_restore(const void* src, int num_src_rows, const int32_t* idx_dev, int rows,
               int64_t row_bytes, void* dst, int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Test hook for the failure path of the attention pipeline (no counterpart on
 * the source pages).  Process-wide; affects launches made after the call.
 *   CPATTN_DEBUG_WAIT_LIMIT_NS: time limit of every mbarrier wait inside the
 *     attention kernels, in ns (default 4e9).  value > 0.
 *   CPATTN_DEBUG_WITHHOLD_Q: value != 0 makes the TMA producer skip the query
 *     load, so the MMA thread's wait on it runs out: the kernel then writes
 *     CPATTN_ERR_TIMEOUT to the status word, drains its own copies, frees its
 *     tensor memory and returns (outputs of the affected tiles are not
 *     written).  Nothing traps and no wait is unbounded.  Reset to 0 after use.
 *   CPATTN_DEBUG_NVTX: value != 0 turns on NVTX ranges named after each entry
 *     point that queues device work (pushed for the host call's duration, for
 *     timeline tools); 0 turns them off.  Off by default unless the
 *     environment variable CPATTN_NVTX is set to a non-zero value.
 * Returns CPATTN_OK or CPATTN_ERR_INVALID_ARG. */
#define CPATTN_DEBUG_WAIT_LIMIT_NS 1
#define CPATTN_DEBUG_WITHHOLD_Q 2
#define CPATTN_DEBUG_NVTX 3
int cp_attn_debug(int knob, long long value);

/* Human-readable name of a status code (static string). */
const char* cp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
