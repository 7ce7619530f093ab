/*
 * gqa_decode.h -- C ABI of libgqadecode.so: single-query (decode-step) grouped-query attention
 * over a KV cache on NVIDIA GB300 (sm_103a), with split-KV flash-decode partials merged by
 * log-sum-exp.
 *
 * What is computed (for query row t, query head h; G = n_heads / n_kv_heads):
 *   g = h / G                        the KV head serving h's group    (attention_gqa.metal,
 *                                     cera 0.5.4: one KV head per group of query heads)
 *   s = seq_of[t]                    which sequence's cache the row reads
 *   J = 0 .. kv_len[t]-1             dense decode, or the first min(kv_len[t], budget) entries
 *                                     of ids[t]                        (qsa2.metal, qsa_attn2)
 *   x_j = scale * q[t][h] . K^[s][j][g]
 *   out[t][h] = sum_j softmax(x)_j * V^[s][j][g]      (attention_gqa.metal phases 1-3;
 *                                     flash_attention.metal, cera 0.2.0, in one online pass)
 *   kv_len[t] == 0 (or an empty id list) gives out[t][h] = 0   (flash_attention.metal, the
 *                                     seq_len == 0 guard)
 * K^/V^ are the cache rows dequantised: f16 widened to fp32, or int8 times the f16 scale of its
 * 64-dim group (qsa2.metal, qsa_attn2).
 *
 * Conventions shared by every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller.  The library never allocates,
 *     frees or synchronises; work is enqueued on `stream` (0 = the legacy default stream) and
 *     runs asynchronously.  Calls are thread-safe; gqa_last_error() is per host thread.
 *   - Layouts are dense, row-major, innermost dimension last:
 *       q      [n_tok][n_heads][head_dim]                      fp32
 *       out    [n_tok][n_heads][head_dim]                      fp32
 *       f16 K/V cache   [n_seq][cache_cap][n_kv_heads][head_dim]   IEEE binary16 bit patterns
 *       int8 K/V cache  [n_seq][cache_cap][n_kv_heads][head_dim]   int8
 *       int8 scales     [n_seq][cache_cap][n_kv_heads][head_dim/64] binary16
 *       kv_len [n_tok] int32: positions row t attends to (decode: the sequence length; a causal
 *              prefill row at position p: p + 1 -- flash_attention_tq.metal, cera 0.4.0)
 *       seq_of [n_tok] int32 or NULL (NULL: row t reads sequence t, which needs n_seq >= n_tok)
 *       ids    [n_tok][budget] int32 cell positions or NULL (NULL: dense 0..kv_len[t]-1)
 *       part   [n_tok][n_split][n_heads][head_dim + 2] fp32: unnormalised acc[head_dim], then
 *              the chunk's max score m (natural-log units), then its sum l  (qsa2.metal,
 *              qsa_attn2's partial layout)
 *   - Alignment: q, out, caches, scales and part must be 16-byte aligned (TMA and vector loads).
 *   - Errors: a gqa_status is returned; nothing is launched unless it is GQA_OK.  Data-dependent
 *     faults are never traps: kernels clamp and OR a bit into *err_word (device int32, may be
 *     NULL to ignore them); see GQA_ERR_*.  err_word is not cleared by the library.
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_ABI_VERSION 9

typedef enum gqa_status {
  GQA_OK = 0,
  GQA_EINVAL = 1,       /* null or misaligned pointer, bad size, n_heads % n_kv_heads != 0,
                           head_dim not in {64, 128, 256}, non-finite scale, bad budget */
  GQA_EWORKSPACE = 2,   /* ws is NULL or smaller than attn_decode_workspace_bytes() */
  GQA_EUNSUPPORTED = 3, /* a valid request this build does not serve (group size > 16) */
  GQA_ECUDA = 4         /* a CUDA runtime/driver call failed; gqa_last_error() has the text */
} gqa_status;

/* Bits OR-ed into *err_word by the kernels (device side, never a trap). */
#define GQA_ERR_KVLEN_RANGE 0x1 /* kv_len[t] < 0 or > cache_cap: clamped into [0, cache_cap] */
#define GQA_ERR_ID_RANGE 0x2    /* an id outside [0, kv_len[t]): that cell is skipped */
#define GQA_ERR_SEQ_RANGE 0x4   /* seq_of[t] outside [0, n_seq): the row writes zeros */
#define GQA_ERR_TIMEOUT 0x8     /* a pipeline wait passed its iteration limit; CTA gave up */

/* Kinds for the planner and the workspace query. */
#define GQA_KIND_F16 0
#define GQA_KIND_Q8 1
#define GQA_KIND_TQ 2 /* TurboQuant-compressed caches (attn_decode_tq) */

/* The split plan the decode calls use (exposed so hosts and tests can inspect it). */
typedef struct gqa_plan {
  int chunk;         /* chunked mode: positions (or selected cells) per KV chunk, a multiple of
                        tile; stream-K mode: 0 */
  int n_split;       /* chunked mode: chunks per row at max_kv_len; stream-K mode: CTAs */
  int tile;          /* positions staged in shared memory per pipeline stage */
  int grid_x, grid_y, grid_z; /* launch grid: chunked (n_split, n_kv_heads x head split,
                                 n_tok, or row-group slots when row_group > 1);
                                 stream-K (CTAs, 1, 1) */
  int merge;         /* 1 when rows may be split: partials go to ws and are merged inside the
                        same kernel by whichever CTA finishes a row's KV head last; rows grouped
                        by sequence are merged inside the kernel by the group's chunk CTAs when
                        the grid fits one CTA per SM, else by a second kernel, one warp per
                        (row, head) */
  int streamk;       /* 1: stream-K split (f16 caches): the (row, KV head, position) stream is
                        cut into equal shares, one per CTA of a persistent grid */
  int row_group;     /* rows one CTA serves from a shared K/V tile: > 1 when rows may share a
                        sequence (n_seq < n_tok; f16 caches with head_dim 64 or 128 and group
                        size 1, 2, 4 or 8, or TurboQuant caches with head_dim 64 or 128), else
                        1 */
  size_t ws_bytes;   /* workspace the call needs (0 when merge == 0) */
} gqa_plan;

/*
 * attn_decode_plan -- the split planner (host only; launches nothing, needs no GPU).
 * Rows are cut into equal chunks (qsa2.metal chunks its id list in fixed 32-cell pieces;
 * FORWARD_MSL's split-T decode uses fixed 512-position partial blocks): enough chunks for about
 * one wave of two CTAs per SM at max_kv_len, none longer than 8192 positions (4096 for f16
 * rows longer than 8192; TurboQuant caches: eight CTAs per SM, at most 1792).  With
 * GQA_F16_SPLIT=streamk in the environment, f16 calls with n_tok <= 8192 use the stream-K
 * split instead: a persistent grid of up to two CTAs per SM, each taking an equal share of
 * all rows' KV positions.
 * When rows may share a sequence (n_seq < n_tok) an f16 or TurboQuant call groups the rows of
 * each run of equal seq_of[] values (up to 64 / group size rows) into one CTA that reads each
 * K/V tile once for all of them; the chunks are then sized for the groups rather than the rows.
 * num_sms <= 0 queries the current CUDA device.  budget < 0 means dense (no id list).  n_seq
 * is the number of sequences in the cache, as passed to the decode call.
 * Returns GQA_EINVAL on bad sizes, GQA_EUNSUPPORTED for group sizes > 16.
 */
gqa_status attn_decode_plan(int n_tok, int n_seq, int n_heads, int n_kv_heads, int head_dim,
                            int max_kv_len, int budget, int kind, int num_sms, gqa_plan* plan);

/*
 * attn_decode_workspace_bytes -- bytes of `ws` that attn_decode_f16 (kind GQA_KIND_F16),
 * attn_decode_q8_sel (GQA_KIND_Q8) or attn_decode_tq (GQA_KIND_TQ) needs for these sizes on
 * the current device; 0 when no split is needed or the sizes are invalid.  It is the arrival
 * counters (n_tok * grid_y * 4 bytes, rounded up to 256; grid_y as attn_decode_plan reports
 * it: n_kv_heads times the head split) followed by the partials: chunked mode n_tok * n_split *
 * n_heads * (head_dim + 2) * 4 bytes (rounded up to 256) and n_valid (n_tok * 4 bytes);
 * stream-K mode (CTAs + n_tok * n_kv_heads) * group * (head_dim + 2) * 4 bytes.
 */
size_t attn_decode_workspace_bytes(int n_tok, int n_seq, int n_heads, int n_kv_heads,
                                   int head_dim, int max_kv_len, int budget, int kind);

/*
 * attn_decode_f16 -- decode attention over an f16 K/V cache.
 * Passages: attention_gqa.metal (cera 0.5.4) for the grouped math and the load-once-per-group
 * structure; flash_attention.metal (cera 0.2.0) for the online softmax and the empty-context
 * rule; qsa2.metal (regolith) qsa_attn2 / qsa_merge2 for the split partials and their merge.
 *   q, out        see layouts; out is fully written (zeros for empty rows)
 *   k_cache, v_cache  f16 caches, n_seq * cache_cap * n_kv_heads * head_dim elements each
 *   kv_len        device [n_tok]; seq_of device [n_tok] or NULL
 *   max_kv_len    host upper bound of kv_len[] (sizes the grid; rows longer than it are
 *                 truncated to it and flagged GQA_ERR_KVLEN_RANGE)
 *   scale         multiplies q.k (finite)
 *   ws, ws_bytes  caller scratch of >= attn_decode_workspace_bytes(..., GQA_KIND_F16) bytes,
 *                 16-byte aligned (may be NULL when that figure is 0).  Its first
 *                 ceil(n_tok * grid_y * 4 / 256) * 256 bytes are arrival counters (per row,
 *                 or per row group, and KV head): they must be zero before the first call that
 *                 uses this ws (zero the buffer once after allocating it); every call leaves
 *                 them zero again, so the same ws serves any later call.  The rest holds the
 *                 split partials (see attn_decode_workspace_bytes); it needs no clearing.
 *                 Calls sharing a ws must not overlap on the GPU.
 *   err_word      device int32 or NULL
 */
gqa_status attn_decode_f16(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           float* out, const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                           int n_seq, int n_heads, int n_kv_heads, int head_dim,
                           int64_t cache_cap, int max_kv_len, float scale, void* ws,
                           size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

/*
 * attn_decode_q8_sel -- decode attention over an int8 K/V cache with one f16 scale per 64 dims,
 * visiting either every position (ids == NULL) or the first min(kv_len[t], budget) entries of
 * the row's selected-cell list ids[t][0..budget).
 * Passages: qsa2.metal (regolith), qsa_attn2 / qsa_attn3 (dequantisation, selected width,
 * chunked partials) and qsa_merge2 (merge; its sigmoid output gate is not part of this call).
 *   kq, vq        int8 caches; ksc, vsc binary16 scales (layouts above); head_dim in {64,128,256}
 *   ids, budget   device [n_tok][budget] int32 or NULL; budget >= 1 when ids != NULL
 *   an id outside [0, kv_len[t]) is skipped and flagged GQA_ERR_ID_RANGE
 *   other arguments as attn_decode_f16 (workspace kind GQA_KIND_Q8, same budget)
 */
gqa_status attn_decode_q8_sel(const float* q, const int8_t* kq, const int8_t* vq,
                              const uint16_t* ksc, const uint16_t* vsc, const int32_t* ids,
                              int budget, float* out, const int32_t* kv_len,
                              const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                              int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                              float scale, void* ws, size_t ws_bytes, int32_t* err_word,
                              cudaStream_t stream);

/*
 * attn_decode_q8_sel_sg -- attn_decode_q8_sel with scale_group dims per f16 scale: 64 as above,
 * or 32, the 32-element blocks of FORWARD_MSL's q8 cache (kv_append_q8 / attn_part2_q8), whose
 * scale plane [max_t][row/32] is ksc here ([n_seq][cap][n_kv_heads][head_dim/32] with n_seq = 1;
 * a caller holding quants and scales in one buffer passes buffer + scale_off as ksc).
 *   ksc, vsc aligned to min(16, 2 * head_dim / scale_group) bytes; scale_group not in {32, 64}
 *   gives GQA_EINVAL.  Other arguments as attn_decode_q8_sel.
 */
gqa_status attn_decode_q8_sel_sg(const float* q, const int8_t* kq, const int8_t* vq,
                                 const uint16_t* ksc, const uint16_t* vsc, int scale_group,
                                 const int32_t* ids, int budget, float* out,
                                 const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                                 int n_seq, int n_heads, int n_kv_heads, int head_dim,
                                 int64_t cache_cap, int max_kv_len, float scale, void* ws,
                                 size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

/*
 * attn_select_topk -- the selected-cell id list of attn_decode_q8_sel (qsa2.metal, qsa_topk2).
 * Row t's cells 0..kv_len[t]-1 come in blocks of 4 (the last block holds kv_len[t] % 4 cells);
 * cell c carries the score of its block, block_scores[t * score_stride + c / 4].  The row keeps
 * the `budget` cells with the largest scores, equal scores going to the lower cell, and writes
 * them in ascending order to ids[t][0..budget).  A row with kv_len[t] <= budget keeps every
 * cell: ids[t] = 0, 1, .., kv_len[t]-1, then -1.  Scores are compared through the
 * order-preserving map of fp32 bit patterns to uint32 (negative values: all bits flipped;
 * others: sign bit set), so -0 ranks below +0; page 1 names this map `okey` without defining
 * it.
 *   block_scores  device fp32 [n_tok][score_stride], score_stride >= max_kv_len / 4 + 1
 *   kv_len        device int32 [n_tok]; values outside [0, max_kv_len] are clamped and flagged
 *                 GQA_ERR_KVLEN_RANGE
 *   ids           device int32 [n_tok][budget], fully written; budget >= 1
 */
gqa_status attn_select_topk(const float* block_scores, int64_t score_stride,
                            const int32_t* kv_len, int n_tok, int max_kv_len, int budget,
                            int32_t* ids, int32_t* err_word, cudaStream_t stream);

/*
 * attn_decode_tq -- decode attention over a TurboQuant-compressed cache
 * (flash_attention_tq.metal, cera 0.4.0).  Keys are scored without reconstruction:
 *   x_j = (norm_j * sum_d q_rot[d] c[kidx_j(d)]
 *          + norm_j * rn_j * qjl_scale * sum_d q_jl[d] s_j(d)) * scale
 * (c = the four centroids, kidx = 2-bit indices, s = +-1 from the QJL sign bits); values are
 * accumulated in the rotated basis, vnorm_j c[vidx_j(d)], and the merged row is rotated back:
 * out = signs * H(acc) / sqrt(D), H the Walsh-Hadamard transform in Sylvester order.  The
 * page's precomputed per-head sum of q_jl is formed in the kernel.
 *   q_rot, q_jl   device fp32 [n_tok][n_heads][head_dim]: the query rotated and JL-projected
 *   Caches are head-major, as the page's compressed regions are: each (sequence, KV head)
 *   holds its cache_cap positions contiguously.
 *   k_polar, v_polar  device uint32 [n_seq][n_kv_heads][cache_cap][head_dim/16], 16-byte
 *                 aligned; 16 two-bit indices per word, index k in bits 2k..2k+1
 *   k_jl          device uint32 [n_seq][n_kv_heads][cache_cap][head_dim/32], 16-byte aligned;
 *                 sign bit of dim 32w + k in bit k of word w
 *   k_norms       device uint32 [n_seq][n_kv_heads][cache_cap], 16-byte aligned: f16 norm in
 *                 the low half, f16 residual norm in the high half; v_norms likewise, f16 norm
 *                 low
 *   centroids     HOST fp32 [4]; signs device fp32 [head_dim] (the rotation's sign flips)
 *   head_dim 32, 64 or 128 (the page's set: a power of two, a multiple of 32, at most 128; 32
 *   runs on the CUDA cores), group size <= 16 (else GQA_EUNSUPPORTED; above 8 heads a KV head's
 *   group is served by two CTAs of heads).
 *   Other arguments as attn_decode_f16; the workspace is attn_decode_workspace_bytes(...,
 *   GQA_KIND_TQ), zeroed once like attn_decode_f16's.
 */
gqa_status attn_decode_tq(const float* q_rot, const float* q_jl, const uint32_t* k_polar,
                          const uint32_t* k_jl, const uint32_t* k_norms, const uint32_t* v_polar,
                          const uint32_t* v_norms, const float* centroids, const float* signs,
                          float qjl_scale, float scale, float* out, const int32_t* kv_len,
                          const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                          int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                          void* ws, size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

/*
 * kv_append_q8 -- quantise new K/V rows into the int8 cache (FORWARD_MSL, kv_append_q8, with
 * the 64-dim scale groups of the cache attn_decode_q8_sel reads).  For every 64-dim group of a
 * (position, KV head) row: d = amax|x| / 127, codes q = rint(x / d) clamped to [-127, 127]
 * (all 0 when d = 0), scale = f16(d); the arithmetic is IEEE fp32 (division to nearest, rint to
 * even).  Writes positions t0 .. t0 + n_new - 1 of sequence `seq`.
 *   k_new, v_new  device fp32 [n_new][n_kv_heads][head_dim], 8-byte aligned
 *   kq, vq, ksc, vsc  the int8 cache and its scales (layouts above), n_seq x cache_cap rows
 *   requires 0 <= seq < n_seq and t0 + n_new <= cache_cap; head_dim in {64, 128, 256}
 */
gqa_status kv_append_q8(const float* k_new, const float* v_new, int n_new, int n_kv_heads,
                        int head_dim, int8_t* kq, int8_t* vq, uint16_t* ksc, uint16_t* vsc,
                        int n_seq, int64_t cache_cap, int seq, int t0, cudaStream_t stream);

/*
 * kv_append_q8_sg -- kv_append_q8 with scale_group dims per scale: 64, or 32 as FORWARD_MSL's
 * kv_append_q8 quantises (one simdgroup per 32-element block there; one warp per block here).
 * The scales are [n_seq][cap][n_kv_heads][head_dim / scale_group]; scale_group not in {32, 64}
 * gives GQA_EINVAL.  Other arguments as kv_append_q8.
 */
gqa_status kv_append_q8_sg(const float* k_new, const float* v_new, int n_new, int n_kv_heads,
                           int head_dim, int scale_group, int8_t* kq, int8_t* vq, uint16_t* ksc,
                           uint16_t* vsc, int n_seq, int64_t cache_cap, int seq, int t0,
                           cudaStream_t stream);

/*
 * attn_merge -- log-sum-exp merge of split partials (qsa2.metal, qsa_merge2; FORWARD_MSL's
 * attn_combine is the same merge in exp2 units):
 *   M = max_c m_c,  e_c = exp(m_c - M),  L = sum_c l_c e_c,  out = sum_c acc_c e_c / L
 * over chunks c < n_valid[t] of row t (n_valid device [n_tok], values clamped to [0, n_split]);
 * a row with n_valid 0 (or L == 0) gets zeros.  part as in the layouts, head_dim in {64,128,256}.
 * The pages multiply the merged row by a sigmoid output gate; attn_merge leaves it out (the
 * plain merge) and attn_merge_gated below applies it.
 */
gqa_status attn_merge(const float* part, const int32_t* n_valid, int n_split, int n_tok,
                      int n_heads, int head_dim, float* out, cudaStream_t stream);

/*
 * attn_decode_f16_noalloc -- attn_decode_f16 without a caller-provided workspace.  The pages
 * have no counterpart of this call; it exists for callers that cannot allocate device memory.
 *
 * Who needs it: hosts that own all device memory and hand a plug-in nothing but its input and
 * output buffers -- e.g. a serving runtime that reserves a fixed arena at start-up and forbids
 * any later cudaMalloc, or a foreign-language caller that reaches this library only through the
 * C ABI and has no allocator of its own.  When a row is split into several KV chunks,
 * attn_decode_f16 needs `ws` for the chunk partials; this call takes them from a static
 * __device__ array of GQA_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library instead.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 *
 *   - Arguments, layouts, results and error bits are those of attn_decode_f16.
 *   - Sizes whose workspace (attn_decode_workspace_bytes(..., budget -1, GQA_KIND_F16) with
 *     max_kv_len capped at cache_cap) exceeds GQA_NOALLOC_SCRATCH_BYTES are refused with
 *     GQA_EWORKSPACE before anything launches; gqa_last_error() gives both sizes.
 *   - Every GPU that loads the library holds the array until the process exits.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and caches it; make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's contents.  Its
 *     leading arrival counters (see attn_decode_f16's ws) are zero when the library loads and
 *     every call leaves them zero again; the partials need no clearing, since each call writes
 *     every partial it reads.  Calls whose kernels overlap on the GPU (different streams, or
 *     threads) race on it; serialise them, e.g. on one stream.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (16 << 20)
gqa_status attn_decode_f16_noalloc(const float* q, const uint16_t* k_cache,
                                   const uint16_t* v_cache, float* out, const int32_t* kv_len,
                                   const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                                   int n_kv_heads, int head_dim, int64_t cache_cap,
                                   int max_kv_len, float scale, int32_t* err_word,
                                   cudaStream_t stream);

/*
 * attn_merge_gated -- attn_merge followed by the sigmoid output gate both pages apply after
 * their merge (qsa2.metal, qsa_merge2; FORWARD_MSL, attn_combine):
 *   out[t][h][d] = merge(...)[t][h][d] / (1 + exp(-gate[(t * n_heads + h) * gate_stride + d]))
 * gate: device fp32, 8-byte aligned; gate_stride even and >= head_dim (head_dim for a plain
 * [n_tok][n_heads][head_dim] gate; 2 * head_dim with gate = qfull + head_dim for the pages'
 * per-head [query | gate] pairs).  Other arguments as attn_merge.
 */
gqa_status attn_merge_gated(const float* part, const int32_t* n_valid, int n_split, int n_tok,
                            int n_heads, int head_dim, const float* gate, int64_t gate_stride,
                            float* out, cudaStream_t stream);

/*
 * The decode calls with the sigmoid output gate applied to every output row.  Both model pages
 * end their decode step with it, after the merge: qsa2.metal (regolith) qsa_merge2 and
 * FORWARD_MSL (cherenkov docs) attn_combine multiply the merged row by sigmoid(gate), the gate
 * being the second half of each head's [query | gate] pair.  Here:
 *   out[t][h][d] = attention(t, h)[d] / (1 + exp(-gate[(t * n_heads + h) * gate_stride + d]))
 * whether the row was split (the gate is applied by whichever kernel merges it) or not (by the
 * kernel that writes it); empty rows stay 0.  For TurboQuant caches the gate applies to the
 * row rotated back.
 *   gate          device fp32, 4-byte aligned, not NULL
 *   gate_stride   floats between consecutive (row, head) gate vectors, >= head_dim: head_dim
 *                 for a plain [n_tok][n_heads][head_dim] gate; 2 * head_dim with
 *                 gate = qfull + head_dim for the pages' per-head [query | gate] pairs
 * Other arguments, layouts, workspaces and errors as the ungated call (attn_decode_f16,
 * attn_decode_q8_sel_sg, attn_decode_tq); a bad gate or stride gives GQA_EINVAL.
 */
gqa_status attn_decode_f16_gated(const float* q, const uint16_t* k_cache,
                                 const uint16_t* v_cache, float* out, const int32_t* kv_len,
                                 const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                                 int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                                 float scale, const float* gate, int64_t gate_stride, void* ws,
                                 size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

gqa_status attn_decode_q8_sel_gated(const float* q, const int8_t* kq, const int8_t* vq,
                                    const uint16_t* ksc, const uint16_t* vsc, int scale_group,
                                    const int32_t* ids, int budget, float* out,
                                    const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                                    int n_seq, int n_heads, int n_kv_heads, int head_dim,
                                    int64_t cache_cap, int max_kv_len, float scale,
                                    const float* gate, int64_t gate_stride, void* ws,
                                    size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

gqa_status attn_decode_tq_gated(const float* q_rot, const float* q_jl, const uint32_t* k_polar,
                                const uint32_t* k_jl, const uint32_t* k_norms,
                                const uint32_t* v_polar, const uint32_t* v_norms,
                                const float* centroids, const float* signs, float qjl_scale,
                                float scale, float* out, const int32_t* kv_len,
                                const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                                int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                                const float* gate, int64_t gate_stride, void* ws,
                                size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

/* Human-readable name of a status; static storage. */
const char* gqa_status_string(gqa_status s);

/* Text of the last error on this host thread ("" if none); valid until the next call. */
const char* gqa_last_error(void);

/* GQA_ABI_VERSION of the loaded library. */
int gqa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
