/*
 * Oracle for block-sparse KV-outer attention -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the GPU path
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library; the product path never calls it.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Sources (fw-ai/minimax-kernels README):
 *   - intro paragraph: a query attends only to the 128-token KV blocks it
 *     selected; the KV-outer formulation loads a block once for every query
 *     that selected it -- a reordering of the same sum, so the oracle loops
 *     over queries instead;
 *   - "Quick start": token-major q [Tq,Hq,128]; paged caches
 *     [pages,Hkv,page_size,128] reached through block_tables; selections
 *     [Tq,Hkv,topk] of 128-token logical blocks; cu_seqlens_q; used_kv_lens;
 *     output [Tq,Hq,128] and FP32 lse [Hq,Tq];
 *   - feature list under "Installation": BF16/FP16/FP8 inputs, head dim 128,
 *     pages of 64 or 128 tokens, varlen batches, MHA/GQA/MQA, causal or not.
 * Readings where the pages are silent (scale 1/sqrt(128), natural-log lse of
 * the scaled scores, bottom-right causal alignment pos = L - Tq + i, GQA head
 * h -> kv head h / G, -1 = no block, set semantics for repeated blocks,
 * empty rows -> out 0 and lse -inf, unscaled e4m3fn) are listed in the
 * design notes.
 *
 * All arithmetic is IEEE double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_BF16 = 0, OR_FP16 = 1, OR_FP8_E4M3 = 2, OR_NVFP4 = 3 };

/* status bits shared in meaning (not in code) with the GPU library */
enum {
  OR_FLAG_SEL_RANGE = 1,   /* selection outside [-1, nblk) */
  OR_FLAG_SEL_DUP = 2,     /* a block repeated within one (token, kv-head) row */
  OR_FLAG_CAUSAL_LEN = 8,  /* causal with used_kv_len < Tq of the sequence */
  OR_FLAG_LEN = 16,        /* used_kv_len < 0 or beyond the block-table capacity */
  OR_FLAG_CU = 128         /* cu_seqlens_q not a valid partition of the tokens */
};

/* Planted mistakes, for the test that checks the pins catch them
 * (tests/test_oracle_mutants.py): a build with -DORACLE_MUTANT=n makes
 * mistake n, listed where it is planted; the default build makes none. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(n) (ORACLE_MUTANT == (n))

typedef struct {
  int32_t num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, topk, page_size, num_pages,
      max_pages_per_seq, causal;
  double softmax_scale; /* 0 => 1/sqrt(head_dim) */
  int32_t q_dtype, kv_dtype;
} oracle_problem;

/* ------------------------------------------------------------------ decode
 * Exact decoding of the storage formats, written from the format
 * definitions (IEEE-754 binary16; bfloat16 = upper half of binary32;
 * OCP FP8 E4M3 "fn": bias 7, no infinities, S.1111.111 is NaN). */
static double decode_bf16(uint32_t bits) {
  uint32_t u = (bits & 0xFFFFu) << (MUT(1) ? 15 : 16); /* mutant 1: misplaced bits */
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double decode_fp16(uint32_t bits) {
  uint32_t s = (bits >> 15) & 1u, e = (bits >> 10) & 0x1Fu, m = bits & 0x3FFu;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m/1024 * 2^-14 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
  return s ? -v : v;
}

static double decode_e4m3(uint32_t bits) {
  uint32_t s = (bits >> 7) & 1u, e = (bits >> 3) & 0xFu, m = bits & 0x7u;
  double v;
  if (e == 15 && m == 7)
    return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + (double)m / 8.0, (int)e - (MUT(2) ? 8 : 7)); /* mutant 2: wrong exponent bias */
  return s ? -v : v;
}

/* OCP MX FP4 E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; no
 * infinities or NaN.  E = 0: m * 0.5; E > 0: 2^(E-1) * (1 + m/2); so the
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
static double decode_e2m1(uint32_t bits) {
  uint32_t s = (bits >> 3) & 1u, e = (bits >> 1) & 3u, m = bits & 1u;
  double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)e - (MUT(23) ? 2 : 1)); /* mutant 23: bias 2 */
  return s ? -v : v;
}

double oracle_decode(int32_t dtype, uint32_t bits) {
  switch (dtype) {
    case OR_BF16: return decode_bf16(bits);
    case OR_FP16: return decode_fp16(bits);
    case OR_FP8_E4M3: return decode_e4m3(bits);
    case OR_NVFP4: return decode_e2m1(bits);
    default: return NAN;
  }
}

static double load_elem(const void* base, int32_t dtype, int64_t idx) {
  if (dtype == OR_FP8_E4M3) return decode_e4m3(((const uint8_t*)base)[idx]);
  return oracle_decode(dtype, ((const uint16_t*)base)[idx]);
}

/* NVFP4 KV cache (the MSA summary page, "Highlighted Details", lists NVFP4
 * among the formats of its sparse attention and decoding; the layout and
 * the scaling below are this library's reading):
 *   - each 16 consecutive elements of a row (one position of one kv head)
 *     share an E4M3 scale; element value = e2m1(code) * e4m3(scale), with
 *     no per-tensor scale;
 *   - a (page, kv head) slab of ps positions holds ps rows of D/2 bytes of
 *     codes (element 2i in the low nibble of byte i, 2i + 1 in the high
 *     nibble), then ps rows of D/16 scale bytes (scale j covers elements
 *     16 j .. 16 j + 15); slabs follow each other as [page][kv head].
 * Element `idx` of the row-major view [page][kv head][ps][D] used for the
 * other dtypes: */
static double load_nvfp4(const void* base, int32_t ps, int32_t D, int64_t idx) {
  const int64_t row = idx / D, d = idx % D;
  const int64_t slab = row / ps, pos = row % ps;
  const uint8_t* sb = (const uint8_t*)base + slab * ps * (D / 2 + D / 16);
  const uint8_t byte = sb[pos * (D / 2) + d / 2];
  const uint32_t code = (MUT(22) ? !(d & 1) : (d & 1)) ? (byte >> 4) : (byte & 0xFu); /* mutant 22: nibbles swapped */
  const uint8_t scale = sb[(int64_t)ps * (D / 2) + pos * (D / 16) + d / 16];
  return decode_e2m1(code) * decode_e4m3(scale);
}

/* a K or V element of the paged cache, element idx of [page][kv head][ps][D] */
static double load_kv(const void* base, const oracle_problem* p, int64_t idx) {
  if (p->kv_dtype == OR_NVFP4) return load_nvfp4(base, p->page_size, p->head_dim, idx);
  return load_elem(base, p->kv_dtype, idx);
}

/* sequence of token t: the s with cu[s] <= t < cu[s+1] (linear scan) */
static int32_t seq_of_token(const int64_t* cu, int32_t B, int64_t t) {
  for (int32_t s = 0; s < B; ++s)
    if (cu[s] <= t && t < cu[s + 1]) return s;
  return -1;
}

/* -------------------------------------------------------------- attention */
typedef struct {
  const oracle_problem* p;
  const void *q, *k, *v;
  const int32_t *sel, *bt, *lens;
  const int64_t *cu, *rows;
  int64_t nrows;
  double *out, *lse;
  int64_t next;
  pthread_mutex_t mu;
  int err;
} attn_job;

/* One output row (token t, query head h), straight from the definition:
 *   K = union over selected blocks b of {p : 128 b <= p < min(128 b + 128, L)},
 *       keeping p <= pos(t) when causal;
 *   s_p = scale * q . k_p;  out = sum_p softmax(s)_p v_p;  lse = log sum_p exp(s_p). */
static int attn_row(const attn_job* J, int64_t t, int32_t h, double* out, double* lse_out) {
  const oracle_problem* p = J->p;
  const int32_t D = p->head_dim, Hq = p->num_q_heads, Hkv = p->num_kv_heads;
  const int32_t G = Hq / Hkv, ps = p->page_size;
  const int32_t g = MUT(3) ? h % Hkv : h / G; /* mutant 3: interleaved GQA map */
  const double scale = MUT(4) ? 1.0 : (p->softmax_scale > 0 ? p->softmax_scale : 1.0 / sqrt((double)D));
  /* mutant 4: the scale dropped */
  for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
  *lse_out = -INFINITY;
  int32_t s = seq_of_token(J->cu, p->num_seqs, t);
  if (s < 0) return 0;
  int64_t L = J->lens[s];
  if (L < 0) L = 0;
  if (L > (int64_t)p->max_pages_per_seq * ps) L = (int64_t)p->max_pages_per_seq * ps;
  const int64_t Tq_s = J->cu[s + 1] - J->cu[s];
  const int64_t pos = L - Tq_s + (t - J->cu[s]) - (MUT(5) ? 1 : 0); /* mutant 5: causal offset */
  const int64_t nblk = (L + 127) / 128;

  unsigned char* in_set = (unsigned char*)calloc((size_t)(L > 0 ? L : 1), 1);
  double* qv = (double*)malloc(sizeof(double) * D);
  double* sc = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  if (!in_set || !qv || !sc) {
    free(in_set); free(qv); free(sc);
    return -1;
  }
  for (int32_t k = 0; k < p->topk; ++k) {
    int32_t b = J->sel[(t * Hkv + g) * p->topk + k];
    if (b < 0 || b >= nblk) continue;
    int64_t hi = 128 * (int64_t)b + 128 < L ? 128 * (int64_t)b + 128 : L;
    if (MUT(6) && hi == 128 * (int64_t)b + 128) --hi; /* mutant 6: a block's last key dropped */
    for (int64_t pp = 128 * (int64_t)b; pp < hi; ++pp)
      if (!p->causal || pp <= pos) in_set[pp] = 1;
  }
  for (int32_t d = 0; d < D; ++d) qv[d] = load_elem(J->q, p->q_dtype, (t * Hq + h) * (int64_t)D + d);

  double m = -INFINITY;
  int64_t count = 0;
  for (int64_t pp = 0; pp < L; ++pp) {
    if (!in_set[pp]) continue;
    int32_t page = J->bt[(int64_t)s * p->max_pages_per_seq + (MUT(7) ? pp / 128 : pp / ps)];
    /* mutant 7: the page walk steps by block, not by page */
    if (page < 0 || page >= p->num_pages) {
      free(in_set); free(qv); free(sc);
      return -2;
    }
    int64_t base = MUT(8) ? (((int64_t)page * ps + pp % ps) * Hkv + g) * D /* mutant 8: [page][pos][head] */
                          : (((int64_t)page * Hkv + g) * ps + pp % ps) * D;
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d) dot += qv[d] * load_kv(J->k, p, base + d);
    sc[pp] = scale * dot;
    if (sc[pp] > m) m = sc[pp];
    ++count;
  }
  if (count > 0) {
    double l = 0.0;
    for (int64_t pp = 0; pp < L; ++pp) {
      if (!in_set[pp]) continue;
      int32_t page = J->bt[(int64_t)s * p->max_pages_per_seq + (MUT(7) ? pp / 128 : pp / ps)];
      int64_t base = MUT(8) ? (((int64_t)page * ps + pp % ps) * Hkv + g) * D
                            : (((int64_t)page * Hkv + g) * ps + pp % ps) * D;
      double w = exp(sc[pp] - m);
      l += w;
      for (int32_t d = 0; d < D; ++d) out[d] += w * load_kv(J->v, p, base + d);
    }
    for (int32_t d = 0; d < D; ++d) out[d] /= l;
    *lse_out = m + (MUT(9) ? log2(l) : log(l)); /* mutant 9: lse in base 2 */
  }
  free(in_set); free(qv); free(sc);
  return 0;
}

static void* attn_worker(void* arg) {
  attn_job* J = (attn_job*)arg;
  const int32_t D = J->p->head_dim, Hq = J->p->num_q_heads;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t i = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (i >= J->nrows) break;
    int64_t r = J->rows ? J->rows[i] : i;
    int rc = attn_row(J, r / Hq, (int32_t)(r % Hq), J->out + i * D, J->lse + i);
    if (rc) {
      pthread_mutex_lock(&J->mu);
      J->err = rc;
      pthread_mutex_unlock(&J->mu);
    }
  }
  return NULL;
}

/* Attention for `nrows` rows given as flat indices t*Hq + h (rows == NULL:
 * every row in order).  out: [nrows][head_dim] double; lse: [nrows] double.
 * Returns 0, or -1 (out of memory) / -2 (a needed page id is invalid) /
 * -3 (bad arguments). */
int oracle_attention_rows(const oracle_problem* p, const void* q, const void* k, const void* v,
                          const int32_t* sel, const int32_t* block_tables, const int64_t* cu_seqlens_q,
                          const int32_t* used_kv_lens, const int64_t* rows, int64_t nrows, double* out,
                          double* lse, int32_t nthreads) {
  if (!p || p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads) return -3;
  attn_job J;
  memset(&J, 0, sizeof J);
  J.p = p; J.q = q; J.k = k; J.v = v; J.sel = sel; J.bt = block_tables; J.cu = cu_seqlens_q;
  J.lens = used_kv_lens; J.rows = rows; J.out = out; J.lse = lse;
  J.nrows = rows ? nrows : (int64_t)p->total_q * p->num_q_heads;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.err;
}

/* ---------------------------------------------------------------- combine
 * Merge of n partial results (o_k, lse_k) of disjoint key subsets of one
 * row into the softmax over their union:
 *   M = max lse_k,  w_k = exp(lse_k - M),  out = sum w_k o_k / sum w_k,
 *   lse = M + log sum w_k.
 * Parts with lse = -inf (empty subsets) carry no weight; no part left gives
 * out = 0 and lse = -inf. */
void oracle_combine(int32_t n, int32_t d, const double* o, const double* lse, double* out, double* lse_out) {
  double M = -INFINITY;
  for (int32_t k = 0; k < n; ++k)
    if (lse[k] > M) M = lse[k];
  for (int32_t j = 0; j < d; ++j) out[j] = 0.0;
  if (M == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double W = 0.0;
  for (int32_t k = 0; k < n; ++k) {
    if (lse[k] == -INFINITY) continue;
    double w = MUT(10) ? 1.0 : exp(lse[k] - M); /* mutant 10: parts averaged unweighted */
    W += w;
    for (int32_t j = 0; j < d; ++j) out[j] += w * o[(int64_t)k * d + j];
  }
  for (int32_t j = 0; j < d; ++j) out[j] /= W;
  *lse_out = M + log(W);
}

/* ------------------------------------------------------------ block index
 * The inverted index of the KV-outer formulation ("loads a selected KV
 * block once and processes all queries that selected it"): for every
 * (kv head g, sequence s, block b) the ordered list of the selection slots
 * that chose it.
 *
 * Definition (exact, integer):
 *   nblk_s  = ceil(L_s / 128) with L_s clamped to [0, max_pages * page_size];
 *   blk_off = exclusive prefix sum of nblk;  NB = sum nblk;
 *   slot    = (t * Hkv + g) * topk + k, taken in increasing order (none
 *             when cu_seqlens_q is not a non-decreasing partition of
 *             [0, total_q]: flag 128, nothing indexed);
 *   a slot is an entry unless its block is -1, out of [0, nblk_s) (flag 1),
 *   equal to an earlier slot's block in the same (t, g) row (flag 2), or,
 *   when causal, starts after the token's position (128 b > pos(t));
 *   key(slot) = g * NB + blk_off[s] + b;
 *   entries   = entry slots sorted by (key, slot);  row_ptr = CSR offsets
 *               over the Hkv * NB keys;  slot_entry[slot] = position or -1.
 * Outputs: row_ptr[Hkv*NB + 1] (capacity row_ptr_cap), entries[nnz],
 * slot_entry[total_q*Hkv*topk].  Returns 0, or -1 (capacity / memory). */
typedef struct {
  int64_t key;
  int64_t slot;
} key_slot;

static int cmp_key_slot(const void* a, const void* b) {
  const key_slot* x = (const key_slot*)a;
  const key_slot* y = (const key_slot*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  if (x->slot != y->slot) return (x->slot < y->slot) != MUT(12) ? -1 : 1; /* mutant 12: slots descending */
  return 0;
}

int oracle_build_index(const oracle_problem* p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                       int32_t* nb_out, int32_t* row_ptr, int64_t row_ptr_cap, int32_t* entries,
                       int32_t* slot_entry, int32_t* nnz_out, int32_t* flags_out) {
  const int32_t B = p->num_seqs, Hkv = p->num_kv_heads, K = p->topk;
  const int64_t cap_len = (int64_t)p->max_pages_per_seq * p->page_size;
  int32_t flags = 0;
  int64_t* nblk = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t* blk_off = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  const int64_t nslots = (int64_t)p->total_q * Hkv * K;
  key_slot* ks = (key_slot*)malloc(sizeof(key_slot) * (size_t)(nslots > 0 ? nslots : 1));
  if (!nblk || !blk_off || !ks) {
    free(nblk); free(blk_off); free(ks);
    return -1;
  }
  if (cu[0] != 0 || cu[B] != p->total_q) flags |= OR_FLAG_CU;
  for (int32_t s = 0; s < B; ++s)
    if (cu[s + 1] < cu[s]) flags |= OR_FLAG_CU;
  int64_t NB = 0;
  for (int32_t s = 0; s < B; ++s) {
    int64_t L = lens[s];
    if (L < 0 || L > cap_len) flags |= OR_FLAG_LEN;
    if (L < 0) L = 0;
    if (L > cap_len) L = cap_len;
    if (p->causal && L < cu[s + 1] - cu[s]) flags |= OR_FLAG_CAUSAL_LEN;
    nblk[s] = (L + 127) / 128;
    blk_off[s] = NB;
    NB += nblk[s];
  }
  const int64_t nkeys = (int64_t)Hkv * NB;
  if (nkeys + 1 > row_ptr_cap) {
    free(nblk); free(blk_off); free(ks);
    return -1;
  }
  int64_t n = 0;
  for (int64_t slot = 0; slot < nslots; ++slot) slot_entry[slot] = -1;
  /* an invalid cu_seqlens_q defines no token -> sequence map: nothing is indexed */
  const int64_t t_end = (flags & OR_FLAG_CU) ? 0 : p->total_q;
  for (int64_t t = 0; t < t_end; ++t) {
    int32_t s = seq_of_token(cu, B, t);
    for (int32_t g = 0; g < Hkv; ++g) {
      for (int32_t k = 0; k < K; ++k) {
        int64_t slot = (t * Hkv + g) * K + k;
        int32_t b = sel[slot];
        if (b == -1 || s < 0) continue;
        if (b < -1 || b >= nblk[s]) {
          flags |= OR_FLAG_SEL_RANGE;
          continue;
        }
        int dup = 0;
        for (int32_t k2 = 0; k2 < k; ++k2)
          if (sel[(t * Hkv + g) * K + k2] == b) dup = 1;
        if (dup) {
          flags |= OR_FLAG_SEL_DUP;
          continue;
        }
        if (p->causal) {
          int64_t L = lens[s] < 0 ? 0 : (lens[s] > cap_len ? cap_len : lens[s]);
          int64_t pos = L - (cu[s + 1] - cu[s]) + (t - cu[s]);
          if (128 * (int64_t)b > pos - (MUT(11) ? 1 : 0)) continue; /* mutant 11: causal drop off by one */
        }
        ks[n].key = g * NB + blk_off[s] + b;
        ks[n].slot = slot;
        ++n;
      }
    }
  }
  qsort(ks, (size_t)n, sizeof(key_slot), cmp_key_slot);
  for (int64_t key = 0; key <= nkeys; ++key) row_ptr[key] = 0;
  for (int64_t i = 0; i < n; ++i) row_ptr[ks[i].key + 1] += 1;
  for (int64_t key = 0; key < nkeys; ++key) row_ptr[key + 1] += row_ptr[key];
  for (int64_t i = 0; i < n; ++i) {
    entries[i] = (int32_t)ks[i].slot;
    slot_entry[ks[i].slot] = (int32_t)i;
  }
  *nb_out = (int32_t)NB;
  *nnz_out = (int32_t)n;
  *flags_out = flags;
  free(nblk); free(blk_off); free(ks);
  return 0;
}

/* ------------------------------------------- block index, physical dedup
 * The index of cross-sequence block dedup: sequences that share a cached
 * prefix point their block tables at the same physical pages, and such a
 * block should be loaded once for every row of every sequence that selected
 * it, not once per sequence.  The block identity becomes physical:
 *
 *   a block (s, b) is SHAREABLE when it is full (128 b + 128 <= L_s) and
 *   its pages are valid: for page_size 128 the page block_tables[s][b], for
 *   64 the pair block_tables[s][2b], [2b+1], each in [0, num_pages);
 *   owner(s, b) = the smallest s' with (s', b) shareable and the same pages
 *   at the same logical block b (s itself when none is smaller); a block
 *   that is not shareable is its own owner;
 *   key(slot)   = g * NB + blk_off[owner(s, b)] + b.
 *
 * Everything else is the plain index's definition above (entries by
 * (key, slot), flags, capacities).  Two sequences' rows meet in one key only
 * for the same logical block of the same physical pages, so the keys, the
 * positions 128 b + i and the valid count 128 agree for every row of the
 * key; each row keeps its own sequence's causal position.  Keys that lost
 * their rows to an owner hold no entries. */
typedef struct {
  int64_t b, page0, page1;
  int32_t s;
} phys_block;

static int cmp_phys_block(const void* a, const void* b) {
  const phys_block* x = (const phys_block*)a;
  const phys_block* y = (const phys_block*)b;
  if (x->b != y->b) return x->b < y->b ? -1 : 1;
  if (x->page0 != y->page0) return x->page0 < y->page0 ? -1 : 1;
  if (x->page1 != y->page1) return x->page1 < y->page1 ? -1 : 1;
  if (x->s != y->s) return x->s < y->s ? -1 : 1;
  return 0;
}

/* owner of every (s, b) at owner[blk_off[s] + b]: the shareable blocks
 * sorted by (b, pages, s); the first of each run of equal (b, pages) owns
 * the run; a block that is not shareable owns itself.  Returns 0 or -1. */
static int fill_owners(const oracle_problem* p, int32_t B, const int64_t* Lc, const int64_t* nblk,
                       const int64_t* blk_off, int64_t NB, const int32_t* block_tables, int32_t* owner) {
  const int32_t ps = p->page_size;
  phys_block* pb = (phys_block*)malloc(sizeof(phys_block) * (size_t)(NB > 0 ? NB : 1));
  if (!pb) return -1;
  int64_t npb = 0;
  for (int32_t s = 0; s < B; ++s) {
    for (int64_t b = 0; b < nblk[s]; ++b) {
      owner[blk_off[s] + b] = s;
      if (128 * b + 128 > Lc[s] && !MUT(13)) continue; /* partial block: never shared (mutant 13: shared) */
      const int32_t* bt = block_tables + (int64_t)s * p->max_pages_per_seq;
      int64_t pg0 = ps == 128 ? bt[b] : bt[2 * b];
      int64_t pg1 = ps == 128 ? -1 : bt[2 * b + 1];
      if (pg0 < 0 || pg0 >= p->num_pages) continue;
      if (ps != 128 && (pg1 < 0 || pg1 >= p->num_pages)) continue;
      pb[npb].b = b;
      pb[npb].page0 = pg0;
      pb[npb].page1 = pg1;
      pb[npb].s = s;
      ++npb;
    }
  }
  qsort(pb, (size_t)npb, sizeof(phys_block), cmp_phys_block);
  for (int64_t i = 0; i < npb; ++i) {
    int64_t first = i;
    while (first > 0 && pb[first - 1].b == pb[i].b && pb[first - 1].page0 == pb[i].page0 &&
           pb[first - 1].page1 == pb[i].page1)
      --first;
    owner[blk_off[pb[i].s] + pb[i].b] = MUT(14) ? pb[i].s : pb[first].s; /* mutant 14: nothing merged */
  }
  free(pb);
  return 0;
}

int oracle_build_index_dedup(const oracle_problem* p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                             const int32_t* block_tables, int32_t* nb_out, int32_t* row_ptr, int64_t row_ptr_cap,
                             int32_t* entries, int32_t* slot_entry, int32_t* nnz_out, int32_t* flags_out) {
  const int32_t B = p->num_seqs, Hkv = p->num_kv_heads, K = p->topk, ps = p->page_size;
  const int64_t cap_len = (int64_t)p->max_pages_per_seq * ps;
  int32_t flags = 0;
  int64_t* nblk = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t* blk_off = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t* Lc = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  const int64_t nslots = (int64_t)p->total_q * Hkv * K;
  key_slot* ks = (key_slot*)malloc(sizeof(key_slot) * (size_t)(nslots > 0 ? nslots : 1));
  if (!nblk || !blk_off || !Lc || !ks) {
    free(nblk); free(blk_off); free(Lc); free(ks);
    return -1;
  }
  if (cu[0] != 0 || cu[B] != p->total_q) flags |= OR_FLAG_CU;
  for (int32_t s = 0; s < B; ++s)
    if (cu[s + 1] < cu[s]) flags |= OR_FLAG_CU;
  int64_t NB = 0;
  for (int32_t s = 0; s < B; ++s) {
    int64_t L = lens[s];
    if (L < 0 || L > cap_len) flags |= OR_FLAG_LEN;
    if (L < 0) L = 0;
    if (L > cap_len) L = cap_len;
    if (p->causal && L < cu[s + 1] - cu[s]) flags |= OR_FLAG_CAUSAL_LEN;
    Lc[s] = L;
    nblk[s] = (L + 127) / 128;
    blk_off[s] = NB;
    NB += nblk[s];
  }
  const int64_t nkeys = (int64_t)Hkv * NB;
  int32_t* owner = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NB > 0 ? NB : 1));
  if (nkeys + 1 > row_ptr_cap || !owner || fill_owners(p, B, Lc, nblk, blk_off, NB, block_tables, owner) != 0) {
    free(nblk); free(blk_off); free(Lc); free(ks); free(owner);
    return -1;
  }
  int64_t n = 0;
  for (int64_t slot = 0; slot < nslots; ++slot) slot_entry[slot] = -1;
  const int64_t t_end = (flags & OR_FLAG_CU) ? 0 : p->total_q;
  for (int64_t t = 0; t < t_end; ++t) {
    int32_t s = seq_of_token(cu, B, t);
    for (int32_t g = 0; g < Hkv; ++g) {
      for (int32_t k = 0; k < K; ++k) {
        int64_t slot = (t * Hkv + g) * K + k;
        int32_t b = sel[slot];
        if (b == -1 || s < 0) continue;
        if (b < -1 || b >= nblk[s]) {
          flags |= OR_FLAG_SEL_RANGE;
          continue;
        }
        int dup = 0;
        for (int32_t k2 = 0; k2 < k; ++k2)
          if (sel[(t * Hkv + g) * K + k2] == b) dup = 1;
        if (dup) {
          flags |= OR_FLAG_SEL_DUP;
          continue;
        }
        if (p->causal) {
          int64_t pos = Lc[s] - (cu[s + 1] - cu[s]) + (t - cu[s]);
          if (128 * (int64_t)b > pos) continue;
        }
        ks[n].key = g * NB + blk_off[owner[blk_off[s] + b]] + b;
        ks[n].slot = slot;
        ++n;
      }
    }
  }
  qsort(ks, (size_t)n, sizeof(key_slot), cmp_key_slot);
  for (int64_t key = 0; key <= nkeys; ++key) row_ptr[key] = 0;
  for (int64_t i = 0; i < n; ++i) row_ptr[ks[i].key + 1] += 1;
  for (int64_t key = 0; key < nkeys; ++key) row_ptr[key + 1] += row_ptr[key];
  for (int64_t i = 0; i < n; ++i) {
    entries[i] = (int32_t)ks[i].slot;
    slot_entry[ks[i].slot] = (int32_t)i;
  }
  *nb_out = (int32_t)NB;
  *nnz_out = (int32_t)n;
  *flags_out = flags;
  free(nblk); free(blk_off); free(Lc); free(ks); free(owner);
  return 0;
}

/* The owner of every block, in key order (sequence s's blocks at
 * blk_off[s] ..): owner_out[NB], NB = sum ceil(L_s / 128) with L_s clamped
 * as above (capacity owner_cap).  Returns NB, or -1 (capacity / memory). */
int64_t oracle_block_owners(const oracle_problem* p, const int32_t* lens, const int32_t* block_tables,
                            int32_t* owner_out, int64_t owner_cap) {
  const int32_t B = p->num_seqs;
  const int64_t cap_len = (int64_t)p->max_pages_per_seq * p->page_size;
  int64_t* nblk = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t* blk_off = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  int64_t* Lc = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
  if (!nblk || !blk_off || !Lc) {
    free(nblk); free(blk_off); free(Lc);
    return -1;
  }
  int64_t NB = 0;
  for (int32_t s = 0; s < B; ++s) {
    int64_t L = lens[s] < 0 ? 0 : (lens[s] > cap_len ? cap_len : lens[s]);
    Lc[s] = L;
    nblk[s] = (L + 127) / 128;
    blk_off[s] = NB;
    NB += nblk[s];
  }
  int64_t rc = NB;
  if (NB > owner_cap || fill_owners(p, B, Lc, nblk, blk_off, NB, block_tables, owner_out) != 0) rc = -1;
  free(nblk); free(blk_off); free(Lc);
  return rc;
}

/* ---------------------------------------------------- top-k block selection
 * The step before the index: which 128-token blocks each (token, kv head)
 * row attends to.  The MSA summary page ("How It Works") names "sparse
 * top-k selection"; the sglang pull request ("Summary") writes an index K
 * cache beside K and V.  The scoring rule itself is not on the pages; this
 * is the library's reading (also in the design notes):
 *   - index query iq[t][g][0..D) and an index key at every cached position p
 *     of the sequence, ik_cache[block_tables[s][p / ps]][g][p % ps][0..D)
 *     (one index head per kv head), both in the problem's kv dtype;
 *   - dot(t, g, p) = the FP32 sum of iq[t][g][d] * ik[p][g][d], accumulated
 *     by fused multiply-add in the order d = 0, 1, .., D-1 starting from +0:
 *     the kernel's precision, since the selection is an integer decision
 *     both sides must take in the same arithmetic;
 *   - score(t, g, b) = the largest dot(t, g, p) over the block's visible
 *     positions: 128 b <= p < min(128 b + 128, L), p <= pos(t) when causal,
 *     and p on a valid page; NaN dots are skipped; a block with no such p
 *     has no score;
 *   - sel[t][g][:] = the blocks that have a score, by score descending and
 *     then block ascending (+0 and -0 are equal), the first topk of them;
 *     the remaining slots are -1.  Tokens outside every sequence get -1. */
typedef struct {
  const oracle_problem* p;
  int32_t dim;
  const void *iq, *ik;
  const int32_t *bt, *lens;
  const int64_t* cu;
  int32_t* sel;
  float* score;
  int64_t max_blocks;
  const int64_t* rows; /* (token * Hkv + kv head) rows to compute, or NULL for all */
  int64_t nrows;
  int64_t next;
  pthread_mutex_t mu;
  int err;
} select_job;

typedef struct {
  float score;
  int32_t b;
} block_score;

static int cmp_block_score(const void* a, const void* b) {
  const block_score* x = (const block_score*)a;
  const block_score* y = (const block_score*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  if (MUT(17)) return x->b > y->b ? -1 : (x->b < y->b ? 1 : 0); /* mutant 17: ties to the larger block */
  return x->b < y->b ? -1 : (x->b > y->b ? 1 : 0);
}

static int select_row(const select_job* J, int64_t t, int32_t g) {
  const oracle_problem* p = J->p;
  const int32_t Hkv = p->num_kv_heads, K = p->topk, ps = p->page_size, D = J->dim;
  int32_t* out = J->sel + (t * Hkv + g) * K;
  for (int32_t k = 0; k < K; ++k) out[k] = -1;
  const int32_t s = seq_of_token(J->cu, p->num_seqs, t);
  if (s < 0) return 0;
  const int64_t cap = (int64_t)p->max_pages_per_seq * ps;
  int64_t L = J->lens[s];
  if (L < 0) L = 0;
  if (L > cap) L = cap;
  const int64_t tq = J->cu[s + 1] - J->cu[s], pos = L - tq + (t - J->cu[s]);
  const int64_t nblk = (L + 127) / 128;
  float* qf = (float*)malloc(sizeof(float) * (size_t)D);
  block_score* bs = (block_score*)malloc(sizeof(block_score) * (size_t)(nblk > 0 ? nblk : 1));
  if (!qf || !bs) {
    free(qf);
    free(bs);
    return -1;
  }
  for (int32_t d = 0; d < D; ++d) qf[d] = (float)load_elem(J->iq, p->kv_dtype, (t * Hkv + g) * D + d);
  int64_t n = 0;
  for (int64_t b = 0; b < nblk; ++b) {
    int have = 0;
    float best = 0.f;
    for (int64_t pp = 128 * b; pp < 128 * b + 128 && pp < L; ++pp) {
      if (p->causal && pp > pos - (MUT(18) ? 1 : 0)) break; /* mutant 18: the row's own position hidden */
      const int32_t page = J->bt[(int64_t)s * p->max_pages_per_seq + pp / ps];
      if (page < 0 || page >= p->num_pages) continue;
      const int64_t base = (((int64_t)page * Hkv + g) * ps + pp % ps) * D;
      float acc = 0.f;
      for (int32_t d = 0; d < D - (MUT(19) ? 1 : 0); ++d) /* mutant 19: the last dimension dropped */
        acc = fmaf(qf[d], (float)load_elem(J->ik, p->kv_dtype, base + d), acc);
      if (isnan(acc)) continue;
      if (!have || (MUT(20) ? acc < best : acc > best)) best = acc; /* mutant 20: the block's minimum */
      have = 1;
    }
    if (J->score && b < J->max_blocks) J->score[(t * Hkv + g) * J->max_blocks + b] = have ? best : NAN;
    if (!have) continue;
    bs[n].score = best == 0.f ? 0.f : best; /* -0 ranks as +0 */
    bs[n].b = (int32_t)b;
    ++n;
  }
  qsort(bs, (size_t)n, sizeof(block_score), cmp_block_score);
  for (int64_t k = 0; k < n && k < K; ++k) out[k] = bs[k].b;
  free(qf);
  free(bs);
  return 0;
}

static void* select_worker(void* arg) {
  select_job* J = (select_job*)arg;
  const int64_t rows = J->rows ? J->nrows : (int64_t)J->p->total_q * J->p->num_kv_heads;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    const int64_t i = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (i >= rows) break;
    const int64_t r = J->rows ? J->rows[i] : i;
    if (select_row(J, r / J->p->num_kv_heads, (int32_t)(r % J->p->num_kv_heads)) != 0) {
      pthread_mutex_lock(&J->mu);
      J->err = 1;
      pthread_mutex_unlock(&J->mu);
    }
  }
  return NULL;
}

/* sel_out int32 [total_q][Hkv][topk]; score_out (may be NULL) float
 * [total_q][Hkv][max_blocks]: each block's score, NaN where it has none.
 * rows (may be NULL): only these (token * Hkv + kv head) rows are computed.
 * Returns 0, or -1 (memory). */
int oracle_select_blocks(const oracle_problem* p, int32_t dim, const void* iq, const void* ik_cache,
                         const int32_t* block_tables, const int64_t* cu, const int32_t* lens, int32_t* sel_out,
                         float* score_out, int64_t max_blocks, const int64_t* rows, int64_t nrows,
                         int32_t nthreads) {
  if (p->kv_dtype == OR_NVFP4) return -2; /* index keys are 16-bit or FP8 */
  select_job J;
  memset(&J, 0, sizeof(J));
  J.p = p;
  J.dim = dim;
  J.iq = iq;
  J.ik = ik_cache;
  J.bt = block_tables;
  J.lens = lens;
  J.cu = cu;
  J.sel = sel_out;
  J.score = score_out;
  J.max_blocks = max_blocks;
  J.rows = rows;
  J.nrows = nrows;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 0; i < nthreads; ++i)
    if (pthread_create(&th[i], NULL, select_worker, &J) == 0) ++started;
  if (started == 0) select_worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.err ? -1 : 0;
}

/* --------------------------------------------------------------- schedule
 * Load-balancing schedule over the index ("load-balancing scheduler" in the
 * README's test list; the splitting rule, the decode merge and the cost
 * model are this library's).
 *
 * Definition (exact, integer), keys with cnt > 0 taken in key order:
 *   G = Hq / Hkv;  a key (g, s, b) is a DECODE key when the sequence has
 *   exactly one new token (Tq_s == 1), G <= 16, and the key holds exactly
 *   one entry, whose token is that one token of s; otherwise it is NORMAL.
 *   (In the plain index every key of such a sequence is a decode key; in
 *   the deduplicated index a key owned by s may hold other sequences'
 *   entries, or none of its own, and is then NORMAL.)
 *   NORMAL: E = rows_per_item_tiles * max(1, 128 / G) entries per item;
 *     n = ceil(cnt / E) items, item i covering entries
 *     [row_ptr[key] + i*cnt/n, row_ptr[key] + (i+1)*cnt/n);
 *     cost = 384 + valid_tokens(key) * kv_weight + tiles * 256 + rows * 3
 *     with tiles = ceil(entries / max(1, 128 / G)), rows = entries * G
 *     (the leading 384 is the item's fixed stage turnover).
 *   DECODE: a run is a maximal sequence of consecutive active decode keys
 *     with the same (g, s) (all hold the same single entry: the one token
 *     of s);
 *     a run of len keys becomes n = ceil(len / decode_blocks) items, item i
 *     covering run positions [i*len/n, (i+1)*len/n);  item = {position of
 *     its first key in the active-key list, entry of that key, 1, nkeys};
 *     cost = sum over its keys of valid_tokens * kv_weight + nkeys * 64 + 256.
 *   valid_tokens = min(128, L_s - 128 b); kv_weight = 2 (16-bit caches) or 1
 *   (FP8 and NVFP4, whose blocks are widened before the MMAs).
 *   Each list (normal, decode) gets its own exclusive cost prefix (total C)
 *   and its own partition: cta_ptr[c] = #{items i : prefix[i] < floor(c*C/P)}.
 * items rows: {key, entry_begin, n_entries, 0} (normal);
 *             {active_pos, entry, 1, nkeys} (decode).
 * out_counts[0] = normal items, out_counts[1] = decode items.
 * Returns 0, or -1 when a capacity is too small. */
static int64_t seq_len_clamped(const oracle_problem* p, const int32_t* lens, int32_t s) {
  const int64_t cap_len = (int64_t)p->max_pages_per_seq * p->page_size;
  return lens[s] < 0 ? 0 : (lens[s] > cap_len ? cap_len : lens[s]);
}

static void key_to_gsb(const oracle_problem* p, const int32_t* lens, int32_t nb, int64_t key, int32_t* g,
                       int32_t* s, int64_t* b) {
  *g = (int32_t)(key / nb);
  int64_t r = key % nb, off = 0;
  int32_t ss;
  for (ss = 0; ss < p->num_seqs; ++ss) {
    int64_t nblk = (seq_len_clamped(p, lens, ss) + 127) / 128;
    if (r < off + nblk) break;
    off += nblk;
  }
  *s = ss;
  *b = r - off;
}

static void partition(int64_t n_items, const int64_t* prefix, int32_t num_ctas, int32_t* cta_ptr) {
  const int64_t C = prefix[n_items];
  for (int32_t c = 0; c <= num_ctas; ++c) {
    int64_t target = (int64_t)c * C / num_ctas, cnt = 0;
    for (int64_t i = 0; i < n_items; ++i)
      if (prefix[i] < target) ++cnt;
    cta_ptr[c] = (int32_t)cnt;
  }
}

/* the decode-key rule above, for the key at active position a */
static int is_decode_key(const oracle_problem* p, const int32_t* lens, const int64_t* cu, int32_t nb,
                         const int32_t* row_ptr, const int32_t* entries, int64_t key) {
  const int32_t G = p->num_q_heads / p->num_kv_heads;
  int32_t g, s;
  int64_t b;
  key_to_gsb(p, lens, nb, key, &g, &s, &b);
  if (cu[s + 1] - cu[s] != 1 || G > 16) return 0;
  if (row_ptr[key + 1] - row_ptr[key] != 1 && !MUT(21)) return 0; /* mutant 21: the entry count ignored */
  const int64_t slot = entries[row_ptr[key]];
  return slot / ((int64_t)p->num_kv_heads * p->topk) == cu[s];
}

int oracle_schedule(const oracle_problem* p, const int32_t* lens, const int64_t* cu, int32_t nb,
                    const int32_t* row_ptr, const int32_t* entries, int32_t rows_per_item_tiles,
                    int32_t decode_blocks, int32_t num_ctas,
                    int32_t* items_n, int64_t* cost_n, int32_t* cta_n, int32_t* items_d, int64_t* cost_d,
                    int32_t* cta_d, int64_t items_cap, int64_t* out_counts) {
  const int32_t Hkv = p->num_kv_heads;
  const int32_t G = p->num_q_heads / Hkv;
  const int32_t per_tile = 128 / G > 0 ? 128 / G : 1;
  const int64_t E = (int64_t)rows_per_item_tiles * per_tile;
  const int32_t kvw = (p->kv_dtype == OR_BF16 || p->kv_dtype == OR_FP16) ? 2 : 1;
  const int64_t nkeys = (int64_t)Hkv * nb;
  /* the active keys, in key order */
  int64_t n_active = 0;
  for (int64_t key = 0; key < nkeys; ++key)
    if (row_ptr[key + 1] > row_ptr[key]) ++n_active;
  int64_t* active = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_active > 0 ? n_active : 1));
  if (!active) return -1;
  n_active = 0;
  for (int64_t key = 0; key < nkeys; ++key)
    if (row_ptr[key + 1] > row_ptr[key]) active[n_active++] = key;
  int64_t nn = 0, nd = 0, Cn = 0, Cd = 0;
  for (int64_t a = 0; a < n_active; ++a) {
    int32_t g, s;
    int64_t b;
    key_to_gsb(p, lens, nb, active[a], &g, &s, &b);
    const int64_t L = seq_len_clamped(p, lens, s);
    const int dec = is_decode_key(p, lens, cu, nb, row_ptr, entries, active[a]);
    if (!dec) {
      const int64_t key = active[a];
      const int64_t cnt = row_ptr[key + 1] - row_ptr[key];
      const int64_t valid = L - 128 * b < 128 ? L - 128 * b : 128;
      const int64_t n = (cnt + E - 1) / E;
      for (int64_t i = 0; i < n; ++i) {
        const int64_t e0 = i * cnt / n, e1 = (i + 1) * cnt / n, ne = e1 - e0;
        if (nn >= items_cap) { free(active); return -1; }
        items_n[4 * nn + 0] = (int32_t)key;
        items_n[4 * nn + 1] = (int32_t)(row_ptr[key] + e0);
        items_n[4 * nn + 2] = (int32_t)ne;
        items_n[4 * nn + 3] = 0;
        cost_n[nn] = Cn;
        Cn += 384 + valid * kvw + ((ne + per_tile - 1) / per_tile) * 256 + ne * G * 3;
        ++nn;
      }
      continue;
    }
    /* decode: only the first key of a run emits; the run ends where (g, s)
       changes or a key that is not a decode key comes */
    if (a > 0 && is_decode_key(p, lens, cu, nb, row_ptr, entries, active[a - 1])) {
      int32_t g2, s2;
      int64_t b2;
      key_to_gsb(p, lens, nb, active[a - 1], &g2, &s2, &b2);
      if (g2 == g && s2 == s) continue;
    }
    int64_t len = 1;
    while (a + len < n_active && is_decode_key(p, lens, cu, nb, row_ptr, entries, active[a + len])) {
      int32_t g2, s2;
      int64_t b2;
      key_to_gsb(p, lens, nb, active[a + len], &g2, &s2, &b2);
      if (g2 != g || s2 != s) break;
      ++len;
    }
    const int64_t n = MUT(15) ? len / decode_blocks + 1 : (len + decode_blocks - 1) / decode_blocks;
    /* mutant 15: one item too many when len is a multiple of decode_blocks */
    for (int64_t i = 0; i < n; ++i) {
      const int64_t k0 = i * len / n, k1 = (i + 1) * len / n;
      if (nd >= items_cap) { free(active); return -1; }
      items_d[4 * nd + 0] = (int32_t)(a + k0);
      items_d[4 * nd + 1] = row_ptr[active[a + k0]];
      items_d[4 * nd + 2] = 1;
      items_d[4 * nd + 3] = (int32_t)(k1 - k0);
      cost_d[nd] = Cd;
      int64_t c = (k1 - k0) * 64 + 256;
      for (int64_t k = k0; k < k1; ++k) {
        int32_t g2, s2;
        int64_t b2;
        key_to_gsb(p, lens, nb, active[a + k], &g2, &s2, &b2);
        c += (L - 128 * b2 < 128 ? L - 128 * b2 : 128) * kvw;
      }
      Cd += c;
      ++nd;
    }
  }
  cost_n[nn] = Cn;
  cost_d[nd] = Cd;
  partition(nn, cost_n, num_ctas, cta_n);
  partition(nd, cost_d, num_ctas, cta_d);
  out_counts[0] = nn;
  out_counts[1] = nd;
  free(active);
  return 0;
}

/* --------------------------------------------------------------- KV store
 * The write side of the paged cache: a sglang pull request on the same
 * pages ("Summary": the fused K/V/index store with an unscaled
 * bf16-to-fp8_e4m3 cast; "Verification": bit-exact against
 * x.float().clamp(-448, 448).to(torch.float8_e4m3fn)).
 *
 * Row (t, h) of a source [n][heads][dim] goes to cache[page][h][off][:] with
 * page = loc[t] / page_size and off = loc[t] % page_size, the slot layout of
 * the paged caches [pages][heads][page_size][dim]; loc[t] < 0 stores nothing
 * for token t.  Into a cache of the source's own dtype the bits are copied;
 * into an e4m3 cache each value is clamped to [-448, 448] and rounded to the
 * nearest e4m3fn value, ties to even (NaN stays NaN with its sign,
 * S.1111.111). */

/* nearest integer to y >= 0, ties to the even one */
static double round_half_even(double y) {
  const double f = floor(y), r = y - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  if (MUT(16)) return f + 1.0; /* mutant 16: ties away from zero */
  return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* e4m3fn: bias 7; exponent field E in 1..15 gives 2^(E-7) * (1 + m/8),
 * E = 0 gives m * 2^-9; E = 15 with m = 7 is NaN, so the largest finite
 * value is 2^8 * 1.75 = 448. */
static uint8_t encode_e4m3(double x) {
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  double a = fabs(x);
  if (a > 448.0) a = 448.0;
  if (a < ldexp(1.0, -6)) {  /* the subnormal range: steps of 2^-9 */
    const double r = round_half_even(a / ldexp(1.0, -9));  /* 0..8; 8 is the smallest normal */
    return (uint8_t)(sign | (uint8_t)r);
  }
  int e2;
  frexp(a, &e2);  /* a = f * 2^e2, f in [0.5, 1) */
  int k = e2 - 1; /* a in [2^k, 2^(k+1)) */
  double r = round_half_even(a / ldexp(1.0, k - 3));  /* 8..16 */
  if (r == 16.0) {
    r = 8.0;
    ++k;
  }
  const int E = k + 7, m = (int)r - 8;
  return (uint8_t)(sign | (uint8_t)(E << 3) | (uint8_t)m);
}

uint32_t oracle_encode_e4m3(double x) { return encode_e4m3(x); }

/* NVFP4 store of one 16-element group (the NVFP4 reading above; the
 * scaling rule is the library's):
 *   amax = the largest |x| over the group's non-NaN elements (0 if none);
 *   scale code = e4m3(amax / 6): the division in IEEE single precision,
 *   then the FP8 store's rounding (clamp to 448, nearest, ties to even);
 *   with sd = the scale's value, an element's code is 0 when sd is 0 or x is
 *   NaN; otherwise the E2M1 value nearest to y = x / sd (single-precision
 *   division), ties to the even mantissa, magnitudes above 6 saturating to
 *   6, with the sign of y. */
static uint8_t encode_e2m1(float y) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const uint8_t sign = signbit(y) ? 8 : 0;
  const double a = fabs((double)y);
  int i = 0;
  while (i < 7) {
    const double mid = 0.5 * (mag[i] + mag[i + 1]);
    if (a < mid) break;
    if (a == mid) {
      if ((i % 2 != 0) != MUT(24)) ++i; /* a tie goes to the even index (mutant 24: to the odd one) */
      break;
    }
    ++i;
  }
  return (uint8_t)(sign | i);
}

static void encode_nvfp4_group(const float* x, uint8_t* codes, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i)
    if (!isnan(x[i]) && fabsf(x[i]) > amax) amax = fabsf(x[i]);
  const float s = amax / (MUT(25) ? 4.0f : 6.0f); /* mutant 25: scaled to 4, not 6 */
  *scale = encode_e4m3((double)s);
  const float sd = (float)decode_e4m3(*scale);
  for (int i = 0; i < 16; ++i) codes[i] = (sd == 0.0f || isnan(x[i])) ? 0 : encode_e2m1(x[i] / sd);
}

uint32_t oracle_encode_e2m1(float y) { return encode_e2m1(y); }

/* Stores n tokens' rows of `src` ([n][heads][dim], dtype src_dtype: bf16 or
 * fp16) into `cache` ([num_pages][heads][page_size][dim], dtype dst_dtype:
 * src_dtype or e4m3).  Returns the number of tokens whose loc lies at or
 * past num_pages * page_size (stored nowhere), or -3 for bad arguments. */
int64_t oracle_store(int32_t src_dtype, int32_t dst_dtype, int64_t n, int32_t heads, int32_t dim,
                     int32_t page_size, int64_t num_pages, const int64_t* loc, const void* src, void* cache) {
  if ((src_dtype != OR_BF16 && src_dtype != OR_FP16) ||
      (dst_dtype != src_dtype && dst_dtype != OR_FP8_E4M3 && dst_dtype != OR_NVFP4) || n < 0 || heads <= 0 ||
      dim <= 0 || page_size <= 0 || num_pages < 0 || (dst_dtype == OR_NVFP4 && dim % 16 != 0))
    return -3;
  int64_t bad = 0;
  for (int64_t t = 0; t < n; ++t) {
    if (loc[t] < 0) continue;
    if (loc[t] >= num_pages * page_size) {
      ++bad;
      continue;
    }
    const int64_t page = loc[t] / page_size, off = loc[t] % page_size;
    if (dst_dtype == OR_NVFP4) {
      /* the slab layout of the NVFP4 reading above */
      for (int32_t h = 0; h < heads; ++h) {
        uint8_t* sb = (uint8_t*)cache + (page * heads + h) * (int64_t)page_size * (dim / 2 + dim / 16);
        for (int32_t j = 0; j < dim / 16; ++j) {
          float x[16];
          uint8_t codes[16], scale;
          for (int i = 0; i < 16; ++i) {
            const uint16_t bits = ((const uint16_t*)src)[(t * heads + h) * dim + 16 * j + i];
            x[i] = (float)(src_dtype == OR_BF16 ? decode_bf16(bits) : decode_fp16(bits));
          }
          encode_nvfp4_group(x, codes, &scale);
          for (int i = 0; i < 16; i += 2)
            sb[off * (dim / 2) + (16 * j + i) / 2] = (uint8_t)(codes[i] | (codes[i + 1] << 4));
          sb[(int64_t)page_size * (dim / 2) + off * (dim / 16) + j] = scale;
        }
      }
      continue;
    }
    for (int32_t h = 0; h < heads; ++h)
      for (int32_t d = 0; d < dim; ++d) {
        const int64_t si = (t * heads + h) * dim + d;
        const int64_t di = ((page * heads + h) * page_size + off) * dim + d;
        const uint16_t bits = ((const uint16_t*)src)[si];
        if (dst_dtype == OR_FP8_E4M3)
          ((uint8_t*)cache)[di] = encode_e4m3(src_dtype == OR_BF16 ? decode_bf16(bits) : decode_fp16(bits));
        else
          ((uint16_t*)cache)[di] = bits;
      }
  }
  return bad;
}
