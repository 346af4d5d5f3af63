/*
 * mxsa -- block-sparse KV-outer attention over a paged KV cache, for one
 * GB300 (sm_103a).  C ABI: plain pointers and sizes, no C++ or torch types.
 *
 * The operation (fw-ai/minimax-kernels README, intro and "Quick start"):
 * every query token t of sequence s attends, per KV head g, only to the
 * 128-token logical KV blocks listed in selected[t, g, :] (-1 = none).  In
 * the KV-outer (KV-stationary) formulation each selected block is loaded
 * from HBM once and used for every (query, GQA query head) row that selected
 * it, producing per-row partial outputs and log-sum-exps that a combine step
 * merges.  The call sequence is
 *
 *     mxsa_build_index -> mxsa_schedule -> mxsa_kvouter_fwd -> mxsa_combine
 *
 * all asynchronous on the caller's CUDA stream, followed optionally by
 * mxsa_read_status.  For token t of sequence s (offset i = t - cu[s]) the
 * result is, with L = used_kv_lens[s], Tq_s = cu[s+1] - cu[s], pos(t) =
 * L - Tq_s + i, G = Hq / Hkv and g = h / G:
 *
 *     K(t,g)   = { p : p in a selected block b (128 b <= p < 128 b + 128),
 *                  p < L, and p <= pos(t) when causal }
 *     s_p      = softmax_scale * q[t,h,:] . k_p
 *     out[t,h] = sum_p softmax(s)_p * v_p            (0 when K(t,g) is empty)
 *     lse[h,t] = log sum_p exp(s_p)   (natural log; -inf when K is empty)
 *
 * Key p lives at k_cache[block_tables[s][p / page_size], g, p % page_size, :].
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer; the library allocates nothing (no
 *     cudaMalloc, no host allocation) and keeps no state between calls.
 *   - "device" pointers must point to GPU memory of the current device;
 *     all must be 16-byte aligned and densely packed in the stated layout.
 *   - Host-side argument errors return synchronously with a status code; the
 *     library never falls back to another implementation silently.
 *   - Data errors found on the device (a selection outside [-1, nblk), a
 *     repeated block in one row, a bad page id, ...) set bits in a status
 *     word inside the index workspace and skip the offending slot or page;
 *     they never trap.  mxsa_read_status returns that word.
 *   - Calls on one workspace set must be ordered on one stream.
 */
#ifndef MXSA_H_
#define MXSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXSA_OK = 0,
  MXSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, inconsistent shape */
  MXSA_ERR_UNSUPPORTED = 2, /* head_dim != 128, page_size not 64/128, G > 128, ... */
  MXSA_ERR_WORKSPACE = 3,   /* a workspace is smaller than mxsa_workspace_size says */
  MXSA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  MXSA_ERR_DATA = 5         /* mxsa_read_status: the device flagged bad input data */
} mxsa_status;

typedef enum { MXSA_BF16 = 0, MXSA_FP16 = 1, MXSA_FP8_E4M3 = 2, MXSA_NVFP4 = 3 } mxsa_dtype;

/* MXSA_NVFP4 caches (the MSA summary page, "Highlighted Details", lists
 * NVFP4 among the formats of sparse attention and decoding; the layout and
 * the scaling are this library's): OCP MX FP4 E2M1 codes, each 16
 * consecutive elements of a row sharing one E4M3 scale (value = e2m1 *
 * scale, no per-tensor scale).  A cache is bytes [num_pages][Hkv][page_size
 * * 72]: per (page, kv head) slab, page_size rows of 64 code bytes (element
 * 2i in the low nibble of byte i, 2i + 1 in the high one) and then
 * page_size rows of 8 scale bytes (scale j for elements 16 j .. 16 j + 15). */

/* Bits of the device status word (mxsa_read_status). */
#define MXSA_FLAG_SEL_RANGE 1   /* selected block outside [-1, ceil(L/128)) : slot ignored */
#define MXSA_FLAG_SEL_DUP 2     /* block repeated in one (token, kv head) row: later slot ignored */
#define MXSA_FLAG_PAGE 4        /* a needed block_tables entry outside [0, num_pages): page skipped */
#define MXSA_FLAG_CAUSAL_LEN 8  /* causal with used_kv_len < new tokens of the sequence */
#define MXSA_FLAG_LEN 16        /* used_kv_len < 0 or > max_pages_per_seq * page_size: clamped */
#define MXSA_FLAG_TIMEOUT 32    /* an on-device wait gave up (result undefined) */
#define MXSA_FLAG_SCHEDULE 64   /* schedule and forward disagree on the CTA count */
#define MXSA_FLAG_CU 128        /* cu_seqlens_q is not a non-decreasing partition of total_q */

/* Problem description (sizes and flags of one call).  The sources: the
 * Quick-start signature and the supported-feature list of the
 * fw-ai/minimax-kernels README. */
typedef struct {
  int32_t num_seqs;          /* B >= 1 */
  int32_t total_q;           /* Tq = cu_seqlens_q[B] >= 0 */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0 and G = Hq / Hkv <= 128 */
  int32_t head_dim;          /* must be 128 */
  int32_t topk;              /* selection slots per (token, kv head), 1..256 */
  int32_t page_size;         /* 64 or 128 tokens */
  int32_t num_pages;         /* physical pages in k_cache / v_cache */
  int32_t max_pages_per_seq; /* row stride of block_tables */
  int32_t causal;            /* 0 or 1 (bottom-right aligned: pos(t) = L - Tq_s + i) */
  float softmax_scale;       /* 0 means 1/sqrt(128) */
  int32_t q_dtype;           /* MXSA_BF16 or MXSA_FP16; the output has this dtype */
  int32_t kv_dtype;          /* q_dtype, MXSA_FP8_E4M3 (unscaled e4m3fn) or MXSA_NVFP4 */
} mxsa_problem;

/* Library version, (major << 16) | minor.  (This library's own; the pages
 * describe no C API.) */
int32_t mxsa_version(void);

/* Human-readable name of a status code (static string).  (This library's
 * own; no passage.) */
const char* mxsa_status_string(mxsa_status status);

/* Workspace sizes (bytes) for a problem.  No passage of the pages defines
 * this call: the README's Quick-start API allocates internally, and this
 * caller-owned-workspace design is the library's own.  Upper bounds computed
 * from the shapes alone (independent of the CTA count: the schedule's
 * per-CTA arrays are sized for MXSA_MAX_CTAS), so one allocation serves
 * any selections / lengths of that shape.  index: inverted block index +
 * device status word; sched: work items and the per-CTA partition; partial:
 * partial outputs and lses, one row of 128 values plus one FP32 lse per
 * (selected block, query head) pair; the rows are FP32 when kv_dtype is
 * MXSA_FP8_E4M3 or MXSA_NVFP4, else in the 16-bit q_dtype.
 * Returns MXSA_ERR_INVALID_ARG / MXSA_ERR_UNSUPPORTED for bad problems. */
mxsa_status mxsa_workspace_size(const mxsa_problem* problem, size_t* index_bytes, size_t* sched_bytes,
                                size_t* partial_bytes);

/* Step 1 -- index builder ("index builder" in the README's test list; the
 * algorithm is this library's): inverts the query -> block selections into
 * block -> (token, head group) lists.  Keys are (kv head g, sequence s,
 * block b) in that order; within a key the entries are the selection slots
 * (t * Hkv + g) * topk + k in increasing t (bit-exact, deterministic).
 *   sel           device int32 [total_q, Hkv, topk], -1 = none
 *   cu_seqlens_q  device int64 [B + 1]
 *   used_kv_lens  device int32 [B]
 *   index_ws      device, index_bytes from mxsa_workspace_size (written)
 * Asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream). */
mxsa_status mxsa_build_index(const mxsa_problem* problem, const int32_t* sel, const int64_t* cu_seqlens_q,
                             const int32_t* used_kv_lens, void* index_ws, size_t index_bytes, void* stream);

/* Step 1, cross-sequence variant.  The README's intro (fw-ai/minimax-kernels)
 * makes the KV block the unit that is loaded once for every query that
 * selected it; with a paged cache, sequences that share a cached prefix
 * point their block_tables at the same physical pages, and this build
 * keys such blocks by the pages, not by the sequence (the rule is this
 * library's reading of that passage):
 *   a block (s, b) is shareable when it is full (128 b + 128 <= L_s) and
 *   its pages (block_tables[s][b] for page_size 128, [2b] and [2b + 1] for
 *   64) lie in [0, num_pages); owner(s, b) = the smallest sequence s' whose
 *   block b is shareable with the same pages (s itself when none is
 *   smaller; a block that is not shareable owns itself); a selection of
 *   (s, b) becomes an entry of key g * NB + blk_off[owner] + b.
 * Everything else is mxsa_build_index's definition: keys (g, s, b) in that
 * order (a key whose rows moved to an owner holds no entries), entries by
 * slot within a key, the same flags and workspace.  A key then holds rows
 * of several sequences; each keeps its own causal position, which the
 * forward reads per row.  mxsa_schedule and mxsa_kvouter_fwd take the
 * result as they take the plain index; mxsa_plan builds the plain index
 * only.
 *   block_tables  device int32 [B, max_pages_per_seq]
 *   dedup_ws      device scratch, dedup_bytes from mxsa_dedup_workspace_size
 *                 (its contents need no initialisation and are not kept)
 * Other arguments as for mxsa_build_index.  Asynchronous on `stream`. */
mxsa_status mxsa_dedup_workspace_size(const mxsa_problem* problem, size_t* dedup_bytes);
mxsa_status mxsa_build_index_dedup(const mxsa_problem* problem, const int32_t* sel, const int64_t* cu_seqlens_q,
                                   const int32_t* used_kv_lens, const int32_t* block_tables, void* index_ws,
                                   size_t index_bytes, void* dedup_ws, size_t dedup_bytes, void* stream);

/* Step 2 -- load-balancing scheduler ("load-balancing scheduler" in the
 * README's test list; the split rule and cost model are this library's):
 * splits each key's entries into work items of at most 4 tiles of 128
 * (token, head) rows and partitions the items into `num_ctas` contiguous
 * ranges of near-equal integer cost.
 *   index_ws   device, written by mxsa_build_index on the same stream
 *   num_ctas   persistent CTAs of the forward; 0 = one per SM of the
 *              current device; at most 4096
 *   sched_ws   device, sched_bytes from mxsa_workspace_size (written) */
mxsa_status mxsa_schedule(const mxsa_problem* problem, const void* index_ws, size_t index_bytes,
                          int32_t num_ctas, void* sched_ws, size_t sched_bytes, void* stream);

/* Steps 1 and 2 in one launch: the same index and schedule as
 * mxsa_build_index followed by mxsa_schedule (bit-identical workspaces),
 * with one kernel launch instead of two.  Arguments as for those calls. */
mxsa_status mxsa_plan(const mxsa_problem* problem, const int32_t* sel, const int64_t* cu_seqlens_q,
                      const int32_t* used_kv_lens, void* index_ws, size_t index_bytes, int32_t num_ctas,
                      void* sched_ws, size_t sched_bytes, void* stream);

/* Step 3 -- KV-outer forward (the README's intro): every work item TMA-loads
 * its KV block (through block_tables) into shared memory once, gathers the
 * q rows of every (token, head) that selected it, and runs q k^T and p v on
 * the tcgen05 tensor cores with FP32 accumulators in tensor memory and the
 * softmax in registers.  Writes one partial row o = sum softmax * v over
 * the block's keys (accumulated in FP32; stored as FP32 with FP8 caches,
 * else rounded to nearest-even in q_dtype: o is a convex combination of V
 * rows, so it stays within their range) and its FP32 lse per (entry, head)
 * into partial_ws.
 *   q             device [total_q, Hq, 128] of q_dtype
 *   k_cache/v_cache device [num_pages, Hkv, page_size, 128] of kv_dtype
 *                 (MXSA_NVFP4: the byte slabs described at mxsa_dtype; FP8
 *                 and NVFP4 blocks are widened exactly to q_dtype before
 *                 the MMAs)
 *   block_tables  device int32 [B, max_pages_per_seq]
 *   num_ctas      must equal the value given to mxsa_schedule (0 = #SMs)
 *   partial_ws    device, partial_bytes from mxsa_workspace_size (written) */
mxsa_status mxsa_kvouter_fwd(const mxsa_problem* problem, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_tables, const void* index_ws,
                             size_t index_bytes, const void* sched_ws, size_t sched_bytes, int32_t num_ctas,
                             void* partial_ws, size_t partial_bytes, void* stream);

/* Step 4 -- combine ("combine" kernel in the README's "Tests" list; output
 * [Tq, Hq, 128] and FP32 lse [Hq, Tq] from its "Quick start"): for each
 * (t, h) merges the partials of the row's selected blocks with LSE weights,
 * in FP32: M = max lse_k, w_k = exp(lse_k - M),
 * out = sum w_k o_k / sum w_k (rounded to nearest-even into q_dtype),
 * lse = M + log sum w_k.  A row with no partial gets out 0 and lse -inf.
 *   out   [total_q, Hq, 128] of q_dtype (written): device memory, or pinned
 *         host memory mapped at the same address (unified addressing), which
 *         the kernel then writes directly over the host link
 *   lse   float [Hq, total_q] (written), same memory rules, or NULL to skip it
 * Pageable host memory or an unknown pointer for out/lse returns
 * MXSA_ERR_INVALID_ARG before any launch. */
mxsa_status mxsa_combine(const mxsa_problem* problem, const void* index_ws, size_t index_bytes,
                         const void* partial_ws, size_t partial_bytes, void* out, float* lse, void* stream);

/* This library's own (no passage; the README's "Backends" section only
 * asks that errors are raised rather than hidden).
 * Synchronises `stream`, then copies the device status word (MXSA_FLAG_*
 * bits) of index_ws into *device_flags.  Returns MXSA_ERR_DATA when any bit
 * is set, MXSA_OK otherwise. */
mxsa_status mxsa_read_status(const void* index_ws, void* stream, int32_t* device_flags);

/* Dense paged attention, the all-blocks-selected case computed directly (no
 * partials, no combine; the MSA project page lists a dense FMHA path next to
 * the sparse one): for token t of sequence s and query head h,
 *   out[t][h][:] = sum_p softmax_p(scale * q[t][h] . k_p) v_p,
 *   lse[h][t] = log sum_p exp(scale * q[t][h] . k_p)   (natural log),
 * over keys p < used_kv_lens[s] (and p <= pos(t) = L - Tq_s + i when causal),
 * k_p / v_p read through block_tables as in mxsa_kvouter_fwd.  No key: out 0,
 * lse -inf.  Same tensors and layouts as the sparse path (q, caches, out
 * [total_q][Hq][128] in q_dtype, lse [Hq][total_q] or NULL); topk is unused
 * and not checked, nor are the sparse index's size limits.
 * kv_dtype must equal q_dtype (BF16/FP16); num_seqs <= 1024.  Tokens outside
 * every sequence (cu_seqlens_q out of order or past total_q) are not written.
 * device_flags (device int32, may be NULL): MXSA_FLAG_PAGE when a needed
 * block_tables entry lies outside [0, num_pages) (that page is skipped and its
 * rows' results are undefined), MXSA_FLAG_TIMEOUT.  Device pointers; q, caches
 * and out 16-byte aligned.  One launch, asynchronous on `stream`;
 * MXSA_ERR_INVALID_ARG / MXSA_ERR_UNSUPPORTED before any launch. */
mxsa_status mxsa_dense_fwd(const mxsa_problem* problem, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int64_t* cu_seqlens_q, const int32_t* used_kv_lens,
                           void* out, float* lse, int32_t* device_flags, void* stream);

/* Paged-cache store, the write side of the caches the forward reads (a
 * sglang pull request on these pages, "Summary": the fused K/V/index store
 * with an unscaled bf16-to-fp8_e4m3 cast).  For each of n_tokens new tokens
 * with slot loc[t] = page * page_size + offset (device int64; loc[t] < 0:
 * token t is not stored):
 *   k_cache[page][h][offset][:] = cast(k[t][h][:]) and likewise v, h < Hkv;
 *   idx_cache[page][j][offset][:] = cast(idx_k[t][j][:]), j < idx_heads.
 * k, v: [n_tokens][num_kv_heads][128] in problem->q_dtype (bf16 or fp16);
 * idx_k: [n_tokens][idx_heads][idx_dim], same dtype, idx_dim a multiple of 8.
 * Of the problem, the store reads the head counts, page size, page count and
 * dtypes; topk, total_q and the sequence fields are not checked.
 * Caches: [num_pages][heads][page_size][dim] in problem->kv_dtype, which is
 * q_dtype (bits copied), MXSA_NVFP4 or MXSA_FP8_E4M3.  MXSA_NVFP4 (the slab
 * layout at mxsa_dtype; no index keys): a group of 16 values stores the
 * scale e4m3(amax / 6) (amax over its non-NaN |x|, single-precision
 * division, rounded as below) and, with sd that scale's value, the E2M1
 * code nearest to x / sd (single precision), ties to even, saturating at
 * 6, with the quotient's sign; NaN elements and groups whose scale is 0
 * store code 0.  MXSA_FP8_E4M3: each value becomes x clamped to
 * [-448, 448] rounded to the nearest e4m3fn value, ties to even, NaN keeping
 * its sign -- bit-identical to x.float().clamp(-448, 448).to(float8_e4m3fn).
 * idx_k and idx_cache are both NULL (no index keys) or both set.
 * device_flags (device int32, may be NULL): MXSA_FLAG_PAGE is ORed in when a
 * slot lies at or past num_pages * page_size (that token is not stored).
 * Device pointers, 16-byte aligned (loc 8-byte); the caller owns all of them.
 * One launch, asynchronous on `stream`.  MXSA_ERR_INVALID_ARG /
 * MXSA_ERR_UNSUPPORTED for bad arguments, before any launch. */
mxsa_status mxsa_store_kv(const mxsa_problem* problem, int64_t n_tokens, const int64_t* loc, const void* k,
                          const void* v, void* k_cache, void* v_cache, const void* idx_k, void* idx_cache,
                          int32_t idx_heads, int32_t idx_dim, int32_t* device_flags, void* stream);

/* Top-k block selection, the step before mxsa_build_index: which 128-token
 * blocks each (token, kv head) row attends to.  The MSA summary page ("How
 * It Works") names the "sparse top-k selection"; the sglang pull request
 * ("Summary") writes an index K cache beside K and V (mxsa_store_kv's
 * idx_cache).  The pages give no scoring rule; this library's reading:
 *   dot(t, g, p)   = the FP32 sum of idx_q[t][g][d] * ik_p[d] over d,
 *                    fused multiply-adds in the order d = 0 .. idx_dim-1
 *                    from +0, where ik_p = idx_cache[block_tables[s][p /
 *                    page_size]][g][p % page_size][:] (one index head per kv
 *                    head); a NaN dot counts as no key;
 *   score(t, g, b) = the largest dot over the block's visible positions:
 *                    128 b <= p < min(128 b + 128, L), p <= pos(t) when
 *                    causal, p on a page in [0, num_pages);
 *   sel[t][g][:]   = the blocks that have a score, by score descending and
 *                    then block ascending (+0 = -0), the first topk of them;
 *                    the remaining slots are -1.
 * The result is exact (bit-identical to a CPU statement of the definition);
 * its rows are valid input for mxsa_plan / mxsa_build_index.
 *   idx_q        device [total_q][Hkv][idx_dim] of kv_dtype (BF16, FP16 or
 *                FP8: an MXSA_NVFP4 problem is MXSA_ERR_UNSUPPORTED)
 *   idx_cache    device [num_pages][Hkv][page_size][idx_dim] of kv_dtype
 *   block_tables, cu_seqlens_q, used_kv_lens as for mxsa_build_index
 *   score_ws     device, score_bytes from mxsa_select_workspace_size: first
 *                the block scores [total_q][Hkv][ceil(max_pages_per_seq *
 *                page_size / 128)] FP32 (NaN: no score), kept for
 *                inspection (entries past a sequence's last block are not
 *                written), then a per-sequence table
 *   sel          device int32 [total_q][Hkv][topk] (written)
 *   device_flags device int32 or NULL: MXSA_FLAG_CU when cu_seqlens_q is not
 *                a non-decreasing partition of total_q (then every row is -1)
 * idx_dim is 64 or 128; num_seqs <= 1024; at most 4096 blocks per sequence.
 * Four launches, asynchronous on `stream`; MXSA_ERR_INVALID_ARG /
 * MXSA_ERR_UNSUPPORTED / MXSA_ERR_WORKSPACE before any launch. */
mxsa_status mxsa_select_workspace_size(const mxsa_problem* problem, int32_t idx_dim, size_t* score_bytes);
mxsa_status mxsa_select_blocks(const mxsa_problem* problem, int32_t idx_dim, const void* idx_q,
                               const void* idx_cache, const int32_t* block_tables, const int64_t* cu_seqlens_q,
                               const int32_t* used_kv_lens, void* score_ws, size_t score_bytes, int32_t* sel,
                               int32_t* device_flags, void* stream);

/* This library's own (no passage).
 * Byte offsets of the arrays inside the index workspace, for inspection
 * (tests compare them bit-exactly with an independent CPU statement).
 * header: int32[16] = {flags, NB (blocks over all sequences), nnz (entries),
 *   n_active (keys with entries), n_keys (Hkv * NB), ...};
 * row_ptr: int32 [n_keys + 1]; entries: int32 [nnz] slot ids;
 * slot_entry: int32 [total_q * Hkv * topk], position in entries or -1;
 * active_keys: int32 [n_active], keys with entries in increasing order. */
typedef struct {
  size_t header, seq_info, token_seq, slot_entry, bitmap, kmap, counts, row_ptr, entries, active_keys,
      active_valid, row_nnz, row_minb, row_maxb, cta_sums, total;
  int64_t keys_cap, nslots, bitmap_words_cap, kmap_bytes_cap, tiles_cap;
} mxsa_index_layout;
mxsa_status mxsa_index_layout_query(const mxsa_problem* problem, mxsa_index_layout* layout);

/* This library's own (no passage).  Byte offsets inside the schedule workspace.  header: int32[16] =
 * {n_items, num_ctas, total cost low, total cost high, (scan counter),
 *  n_dec_items, decode cost low, decode cost high, ...};
 * Two lists, each with int64 exclusive cost prefixes [n + 1] and its own
 * partition cta_ptr int32 [num_ctas + 1]:
 *   items:     int32[4] = {key, entry_begin, n_entries, 0}, keys of
 *              sequences with several new tokens (KV-stationary tiles);
 *   items_dec: int32[4] = {position in active_keys, entry, 1, n_keys}, runs
 *              of up to 8 consecutive decode keys of one sequence and kv
 *              head.  A decode key belongs to a sequence with one new token
 *              (G <= 16) and holds exactly one entry, of that token.  With
 *              the plain index every key of such a sequence is one; with the
 *              dedup index a shared block's key holds several sequences'
 *              entries and goes to the first list.
 * decode_bits: uint32 words, bit a set when active key a is a decode key. */
typedef struct {
  size_t header, items, cost_prefix, cta_ptr, items_dec, cost_prefix_dec, cta_ptr_dec, cta_sums, decode_bits, total;
  int64_t items_cap, tiles_cap;
} mxsa_sched_layout;
mxsa_status mxsa_sched_layout_query(const mxsa_problem* problem, mxsa_sched_layout* layout);

/* The whole call (index, schedule, forward, combine) without any
 * caller-provided workspace.  The pages describe no such entry point; it
 * exists for callers that may not allocate device memory themselves, such as
 * plug-ins of a host runtime that plans every buffer up front, or hot loops
 * that must not risk the device-wide synchronisation a cudaMalloc/cudaFree
 * can cause.  The caller passes inputs and outputs exactly as for the four
 * steps (same layouts and dtypes; lse may be NULL); all scratch lives in one
 * fixed 16 MiB device array inside the library, which every GPU that loads
 * the library keeps reserved until the process exits.  Problems whose three
 * workspaces (mxsa_workspace_size) add up to more than 16 MiB are rejected
 * with MXSA_ERR_WORKSPACE before anything runs.  Nothing is allocated.
 * The first call on a device looks up the array's device address: made
 * while `stream` is being captured it returns MXSA_ERR_INVALID_ARG, as does
 * a stream of another device than the current one (nothing runs).  Calls
 * share the array: calls that overlap on the GPU race and must be
 * serialised by the caller.  Asynchronous on `stream`; the device status
 * word of the last call (data errors, MXSA_FLAG_TIMEOUT) is read with
 * mxsa_noalloc_read_status. */
mxsa_status mxsa_attention_noalloc(const mxsa_problem* problem, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* sel, const int32_t* block_tables,
                                   const int64_t* cu_seqlens_q, const int32_t* used_kv_lens, void* out, float* lse,
                                   void* stream);

/* This library's own (no passage), the companion of mxsa_attention_noalloc:
 * synchronises `stream`, then copies the status word (MXSA_FLAG_* bits) that
 * the last mxsa_attention_noalloc call on the current device left in the
 * library's array into *device_flags.  Returns MXSA_ERR_DATA when any bit
 * is set, MXSA_OK otherwise (MXSA_ERR_INVALID_ARG as for that call). */
mxsa_status mxsa_noalloc_read_status(void* stream, int32_t* device_flags);

/* Rows per tile, tiles per normal work item and blocks per decode work item
 * used by the scheduler. */
#define MXSA_TILE_ROWS 128
#define MXSA_ITEM_TILES 4
#define MXSA_DECODE_BLOCKS 8
#define MXSA_MAX_CTAS 4096

#ifdef __cplusplus
}
#endif
#endif /* MXSA_H_ */
