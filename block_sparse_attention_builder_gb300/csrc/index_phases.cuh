// Device-side phases of the index builder, shared by the index kernel and
// the fused index + schedule kernel.  See index.cu for the algorithm.
#pragma once
#include "internal.h"

namespace mxsa {
namespace ixp {


template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive scan across the CTA (blockDim.x a multiple of 32, <= 1024).
// `tmp` holds 33 elements of shared memory.  Returns the exclusive prefix;
// *total receives the CTA sum.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* tmp, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T inc = warp_inclusive_scan(v);
  if (lane == 31) tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nw ? tmp[lane] : T(0);
    T wi = warp_inclusive_scan(w);
    if (lane < nw) tmp[lane] = wi - w;
    if (lane == nw - 1) tmp[32] = wi;
  }
  __syncthreads();
  T r = tmp[warp] + inc - v;
  *total = tmp[32];
  __syncthreads();
  return r;
}

// Three exclusive scans across the CTA at once (one round of barriers).
// `tmp` holds 3 * 33 elements of shared memory.
struct L3 {
  long long a, b, c;
};
__device__ __forceinline__ L3 block_exclusive_scan3(L3 v, long long* tmp, L3* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const L3 inc{warp_inclusive_scan(v.a), warp_inclusive_scan(v.b), warp_inclusive_scan(v.c)};
  if (lane == 31) {
    tmp[warp] = inc.a;
    tmp[33 + warp] = inc.b;
    tmp[66 + warp] = inc.c;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const long long x = lane < nw ? tmp[33 * j + lane] : 0;
      const long long xi = warp_inclusive_scan(x);
      if (lane < nw) tmp[33 * j + lane] = xi - x;
      if (lane == nw - 1) tmp[33 * j + 32] = xi;
    }
  }
  __syncthreads();
  const L3 r{tmp[warp] + inc.a - v.a, tmp[33 + warp] + inc.b - v.b, tmp[66 + warp] + inc.c - v.c};
  *total = L3{tmp[32], tmp[65], tmp[98]};
  __syncthreads();
  return r;
}

// Totals of the sequence scan (blocks, bitmap words and kmap bytes per kv head).
struct SeqTotals {
  long long nb, bmw, kmw;
};

// Sequence scan over the B sequences by one CTA.  Every CTA that runs it
// gets the totals; only the writer stores seq_info, flags and the header.
// Per-sequence facts a CTA keeps in shared memory (batches of up to
// kSeqTab sequences): block offset, bitmap offset, kmap offset, first
// token, clamped KV length and new tokens.  `find` maps a block row r to
// its sequence (largest s with blk_off <= r) and `get` returns the
// sequence's SeqInfo, from the table when it holds the batch, else from
// global memory.
constexpr int kSeqTab = 512;
struct SeqTab {
  const SeqInfo* g;
  const int (*t)[kSeqTab];
  int B;
  __device__ __forceinline__ bool local() const { return t != nullptr; }
  __device__ __forceinline__ int find(int r) const {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      const int off = local() ? t[0][mid] : g[mid].blk_off;
      if (off <= r) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  }
  __device__ __forceinline__ SeqInfo get(int s) const {
    if (!local()) return g[s];
    SeqInfo si;
    si.blk_off = t[0][s];
    si.bm_off = t[1][s];
    si.km_off = t[2][s];
    si.q_begin = t[3][s];
    si.L = t[4][s];
    si.tq = t[5][s];
    si.nblk = (si.L + 127) / 128;
    si.words = (si.tq + 31) / 32;
    return si;
  }
};

__device__ __forceinline__ SeqTotals phase_seq(const IndexPtrs& ix, const int64_t* cu, const int32_t* lens, int B,
                                               int total_q, int Hkv, int cap_len, int causal, long long* tmp,
                                               bool writer = true, int (*tab)[kSeqTab] = nullptr) {
  long long carry_blk = 0, carry_bm = 0, carry_km = 0;
  int flags = 0;
  // cu_seqlens_q must be a non-decreasing partition of [0, total_q]; if it is
  // not, every sequence is treated as having no new tokens (nothing indexed),
  // which keeps all per-sequence regions inside their shape-derived bounds.
  // The first chunk's lengths load in the same round trip as the check.
  bool bad = threadIdx.x == 0 && (cu[0] != 0 || cu[B] != (int64_t)total_q);
  for (int s = threadIdx.x; s < B; s += blockDim.x) bad |= cu[s + 1] < cu[s];
  const int len0 = (int)threadIdx.x < B ? lens[threadIdx.x] : 0;
  const bool cu_ok = !__syncthreads_or(bad);
  if (!cu_ok) flags |= MXSA_FLAG_CU;
  for (int base = 0; base < B; base += blockDim.x) {
    const int s = base + threadIdx.x;
    long long nblk = 0, bmw = 0, kmw = 0;
    int L = 0, tq = 0, q0 = 0, words = 0;
    if (s < B) {
      const int64_t c0 = cu[s], c1 = cu[s + 1];
      tq = cu_ok ? (int)(c1 - c0) : 0;
      q0 = cu_ok ? (int)c0 : 0;
      const int Lr = base == 0 ? len0 : lens[s];
      if (Lr < 0 || Lr > cap_len) flags |= MXSA_FLAG_LEN;
      L = Lr < 0 ? 0 : (Lr > cap_len ? cap_len : Lr);
      if (causal && L < tq) flags |= MXSA_FLAG_CAUSAL_LEN;
      nblk = (L + 127) / 128;
      words = (tq + 31) / 32;
      bmw = nblk * words;
      kmw = nblk * tq;
    }
    L3 t3;
    const L3 e3 = block_exclusive_scan3(L3{nblk, bmw, kmw}, tmp, &t3);
    if (tab != nullptr && s < B && B <= kSeqTab) {
      tab[0][s] = (int)(carry_blk + e3.a);
      tab[1][s] = (int)(carry_bm + e3.b);
      tab[2][s] = (int)(carry_km + e3.c);
      tab[3][s] = q0;
      tab[4][s] = L;
      tab[5][s] = tq;
    }
    if (s < B && writer) {
      SeqInfo si;
      si.L = L;
      si.nblk = (int)nblk;
      si.blk_off = (int)(carry_blk + e3.a);
      si.tq = tq;
      si.q_begin = q0;
      si.bm_off = (int)(carry_bm + e3.b);
      si.km_off = (int)(carry_km + e3.c);
      si.words = words;
      ix.seq[s] = si;
    }
    carry_blk += t3.a;
    carry_bm += t3.b;
    carry_km += t3.c;
  }
  // OR the per-thread flags together
  int f = __reduce_or_sync(0xffffffffu, flags);
  __shared__ int fl;
  if (threadIdx.x == 0) fl = 0;
  __syncthreads();
  if ((threadIdx.x & 31) == 0 && f) atomicOr(&fl, f);
  __syncthreads();
  if (threadIdx.x == 0 && writer) {
    if (fl) atomicOr(&ix.hdr[kHdrFlags], fl);
    ix.hdr[kHdrNB] = (int)carry_blk;
    ix.hdr[kHdrNnz] = 0;
    ix.hdr[kHdrActive] = 0;
    ix.hdr[kHdrKeys] = (int)(carry_blk * Hkv);
    ix.hdr[kHdrBMW] = (int)carry_bm;
    ix.hdr[kHdrKMW] = (int)carry_km;
    ix.hdr[kHdrTileCtr] = 0;
    ix.row_ptr[0] = 0;
  }
  return SeqTotals{carry_blk, carry_bm, carry_km};
}

__device__ __forceinline__ void phase_zero(const IndexPtrs& ix, int Hkv, const SeqTotals& tot,
                                           bool zero_counts = true) {
  const long long n_keys = tot.nb * Hkv;
  const long long n_bm = tot.bmw * Hkv;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (zero_counts)
    for (long long i = tid; i < n_keys; i += stride) ix.counts[i] = 0;
  for (long long i = tid; i < n_bm; i += stride) ix.bitmap[i] = 0u;
}

// token -> sequence: the last s with cu[s] <= t (sequences of zero tokens
// are skipped naturally).  With `first` (the table's first tokens, B <=
// kSeqTab) the search runs in shared memory; those are cu[s] when
// cu_seqlens_q is valid and all 0 otherwise, when no token has a sequence
// and any s in range will do.
__device__ __forceinline__ void phase_token_seq(const IndexPtrs& ix, const int64_t* cu, int B, int total_q,
                                                const int* first = nullptr) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long t = tid; t < total_q; t += stride) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((first ? (long long)first[mid] : (long long)cu[mid]) <= t) lo = mid;
      else hi = mid - 1;
    }
    ix.token_seq[t] = lo;
  }
}

constexpr int kMarkWarps = 8;
constexpr int kMarkRows = 8;  // most (token, kv head) rows one warp marks per pass

// One warp marks up to kMarkRows consecutive (token, kv head) rows per pass
// (as many as fit 256 selection slots), so the loads of several rows are in
// flight together: the selections of all of them in one coalesced read, the
// sequence facts of row r by lane r.  Lanes then take the pass's slots in
// order; each row's entry count and smallest / largest block are summed over
// the lanes holding its slots.  count = false leaves counts alone (the caller
// derives them from the bitmap rows), so popular blocks cost no contended
// atomics.
__device__ __forceinline__ void phase_mark(const IndexPtrs& ix, const int32_t* sel, int total_q, int Hkv, int topk,
                                           int causal, int32_t (*rowbuf)[256], bool count = true) {
  // per row of the pass: nblk, token index in its sequence (-1: none),
  // causal position, bitmap offset, kmap offset, words, tq, block offset,
  // kv head, then the row's entry count, smallest and largest block
  __shared__ int s_row[kMarkWarps][kMarkRows][12];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const long long n_rows = (long long)total_q * Hkv;
  // rows per pass: enough to give every warp of the grid work, at most
  // kMarkRows and 256 slots (1 <= topk <= 256)
  const long long warps = (long long)gridDim.x * kMarkWarps;
  const int rp = (int)max(1ll, min((long long)min(kMarkRows, 256 / topk), (n_rows + warps - 1) / warps));
  const long long stride = warps * rp;
  int flags = 0;
  for (long long r0 = ((long long)blockIdx.x * kMarkWarps + w) * rp; r0 < n_rows; r0 += stride) {
    const int nr = (int)min((long long)rp, n_rows - r0);
    const int ns = nr * topk;
    const int32_t* srow = sel + r0 * topk;
    for (int x = lane; x < ns; x += 32) rowbuf[w][x] = srow[x];
    if (lane < nr) {
      const long long row = r0 + lane;
      const int t = (int)(row / Hkv), g = (int)(row - (long long)t * Hkv);
      const SeqInfo si = ix.seq[ix.token_seq[t]];
      const int i = t - si.q_begin;
      int* f = s_row[w][lane];
      f[0] = si.nblk;
      f[1] = (i >= 0 && i < si.tq) ? i : -1;
      f[2] = si.L - si.tq + i;
      f[3] = si.bm_off;
      f[4] = si.km_off;
      f[5] = si.words;
      f[6] = si.tq;
      f[7] = si.blk_off;
      f[8] = g;
      f[9] = 0;
      f[10] = 0x7fffffff;
      f[11] = -1;
    }
    __syncwarp();
    for (int x0 = 0; x0 < ns; x0 += 32) {
      const int x = x0 + lane;
      const int r = x < ns ? x / topk : nr;  // nr: past the pass
      const int* f = s_row[w][r < nr ? r : 0];
      const int i = f[1];
      bool cand = false;  // a block of the sequence, for a token of the sequence
      int b = 0;
      if (x < ns) {
        ix.slot_entry[r0 * topk + x] = -1;
        b = rowbuf[w][x];
        if (b != -1 && i >= 0) {
          if (b < -1 || b >= f[0]) flags |= MXSA_FLAG_SEL_RANGE;
          else cand = true;
        }
      }
      // repeated earlier in its row: at a lower lane of this 32-slot step
      // (the lanes with the same row and block), or in an earlier step
      const unsigned long long tag = cand ? ((unsigned long long)r << 32) | (unsigned)b
                                          : (~0ull << 32) | (unsigned)lane;
      const unsigned same = __match_any_sync(0xffffffffu, tag);
      bool ok = false;
      if (cand) {
        bool dup = (same & ((1u << lane) - 1)) != 0;
        for (int k2 = r * topk; k2 < x0; ++k2) dup |= rowbuf[w][k2] == b;
        if (dup) flags |= MXSA_FLAG_SEL_DUP;
        else ok = !(causal && 128 * b > f[2]);  // a block entirely after the token: no entry
      }
      if (ok) {
        const int g = f[8], k = x - r * topk;
        const size_t word = (size_t)g * BMW + (size_t)f[3] + (size_t)b * f[5] + (i >> 5);
        atomicOr(&ix.bitmap[word], 1u << (i & 31));
        ix.kmap[(size_t)g * KMW + (size_t)f[4] + (size_t)b * f[6] + i] = (uint8_t)k;
        if (count) atomicAdd(&ix.counts[(long long)g * NB + f[7] + b], 1);
      }
      // the lanes of each row (the same r) sum their share; the lowest adds it
      const unsigned grp = __match_any_sync(0xffffffffu, r);
      const int made = __reduce_add_sync(grp, ok ? 1 : 0);
      const int bmin = __reduce_min_sync(grp, ok ? b : 0x7fffffff);
      const int bmax = __reduce_max_sync(grp, ok ? b : -1);
      if (r < nr && lane == __ffs(grp) - 1) {
        int* fr = s_row[w][r];
        fr[9] += made;
        fr[10] = min(fr[10], bmin);
        fr[11] = max(fr[11], bmax);
      }
      __syncwarp();
    }
    if (lane < nr) {
      const long long row = r0 + lane;
      const int* f = s_row[w][lane];
      ix.row_nnz[row] = f[9];
      ix.row_minb[row] = f[10];
      ix.row_maxb[row] = f[11];
    }
    __syncwarp();
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(&ix.hdr[kHdrFlags], flags);
}

__device__ __forceinline__ int seq_of_block(const SeqInfo* seq, int B, int r) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (seq[mid].blk_off <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <typename T>
__device__ __forceinline__ T block_sum(T v, T* tmp) {
  T total;
  block_exclusive_scan(v, tmp, &total);
  return total;
}

// Keys are cut into gridDim.x contiguous chunks; CTA c owns chunk c.
__device__ __forceinline__ void key_chunk(int n_keys, int* lo, int* hi) {
  const long long chunk = ((long long)n_keys + gridDim.x - 1) / gridDim.x;
  const long long a = (long long)blockIdx.x * chunk, b = a + chunk;
  *lo = (int)(a < n_keys ? a : n_keys);
  *hi = (int)(b < n_keys ? b : n_keys);
}

// payload of one key in the scans: (entries << 31) | (key has entries)
__device__ __forceinline__ unsigned long long key_payload(int c) {
  return ((unsigned long long)c << 31) | (c > 0 ? 1ull : 0ull);
}

// reduce: per-CTA sum of the payloads of its chunk
__device__ __forceinline__ void phase_key_reduce(const IndexPtrs& ix, unsigned long long* tmp) {
  int lo, hi;
  key_chunk(ix.hdr[kHdrKeys], &lo, &hi);
  unsigned long long v = 0;
  for (int k = lo + threadIdx.x; k < hi; k += blockDim.x) v += key_payload(ix.counts[k]);
  v = block_sum(v, tmp);
  if (threadIdx.x == 0) ix.cta_sums[blockIdx.x] = v;
}

// Writes the entries of the set bits of one bitmap word (word `w` of its
// row: tokens 32 w + bit), starting at entry j; returns the next entry.  The
// bits go in batches of kEmitBatch so that their kmap loads are in flight
// together instead of one dependent load per entry.
constexpr int kEmitBatch = 8;
__device__ __forceinline__ int emit_word(const IndexPtrs& ix, uint32_t bits, int w, const uint8_t* km, int q_begin,
                                         int g, int Hkv, int topk, int j) {
  while (bits) {
    int i[kEmitBatch], k[kEmitBatch];
#pragma unroll
    for (int u = 0; u < kEmitBatch; ++u) {
      i[u] = bits ? w * 32 + __ffs(bits) - 1 : -1;
      bits &= bits - 1;
    }
#pragma unroll
    for (int u = 0; u < kEmitBatch; ++u) k[u] = i[u] >= 0 ? km[i[u]] : 0;
#pragma unroll
    for (int u = 0; u < kEmitBatch; ++u) {
      if (i[u] >= 0) {
        const int slot = ((q_begin + i[u]) * Hkv + g) * topk + k[u];
        ix.entries[j] = slot;
        ix.slot_entry[slot] = j;
        ++j;
      }
    }
  }
  return j;
}

// Writes the entries of one bitmap row: `n_words` words starting at `bm`,
// for tokens q_begin + 32 w + bit.  Serial over the row (one lane).
__device__ __forceinline__ void emit_row_serial(const IndexPtrs& ix, const uint32_t* bm, int n_words,
                                                const uint8_t* km, int q_begin, int g, int Hkv, int topk,
                                                int base) {
  int j = base;
  for (int w = 0; w < n_words; ++w) j = emit_word(ix, bm[w], w, km, q_begin, g, Hkv, topk, j);
}

// One warp writes the entries of a long bitmap row, 32 words at a time
// with a prefix over the words' popcounts.
__device__ __forceinline__ void emit_row_warp(const IndexPtrs& ix, const uint32_t* bm, int n_words,
                                              const uint8_t* km, int q_begin, int g, int Hkv, int topk, int base) {
  const int lane = threadIdx.x & 31;
  int run = base;
  for (int w0 = 0; w0 < n_words; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t bits = w < n_words ? bm[w] : 0u;
    const int cnt = __popc(bits);
    const int inc = warp_inclusive_scan(cnt);
    emit_word(ix, bits, w, km, q_begin, g, Hkv, topk, run + inc - cnt);
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
}

// The same for one of `wcount` warps sharing a long row: warp `wsub` emits
// the row's 32-word chunks wsub, wsub + wcount, ...; the entries before each
// of its chunks are counted from the bitmap words themselves.
__device__ __forceinline__ void emit_row_shared(const IndexPtrs& ix, const uint32_t* bm, int n_words,
                                                const uint8_t* km, int q_begin, int g, int Hkv, int topk, int base,
                                                int wsub, int wcount) {
  const int lane = threadIdx.x & 31;
  int run = base, counted = 0;  // entries of words [0, counted)
  for (int w0 = wsub * 32; w0 < n_words; w0 += wcount * 32) {
    int skip = 0;
    for (int w = counted + lane; w < w0; w += 32) skip += __popc(bm[w]);
    run += __reduce_add_sync(0xffffffffu, skip);
    const int w = w0 + lane;
    const uint32_t bits = w < n_words ? bm[w] : 0u;
    const int cnt = __popc(bits);
    const int inc = warp_inclusive_scan(cnt);
    emit_word(ix, bits, w, km, q_begin, g, Hkv, topk, run + inc - cnt);
    run += __shfl_sync(0xffffffffu, inc, 31);
    counted = w0 + 32 < n_words ? w0 + 32 : n_words;
  }
}

// scan + emit: each CTA adds the sums of the chunks before its own, scans
// its chunk in tiles (row_ptr, the list of keys with entries and their valid
// token counts) and writes the entries of its keys: rows of at most two
// bitmap words one lane per key, longer rows one warp per key.
__device__ __forceinline__ void phase_key_scan_emit(const IndexPtrs& ix, int B, int Hkv, int topk, unsigned long long* tmp) {
  __shared__ int long_key[kScanTile];
  __shared__ int long_base[kScanTile];
  __shared__ int n_long;
  const int n_keys = ix.hdr[kHdrKeys];
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  unsigned long long pre = 0, all = 0;
  for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
    const unsigned long long v = ix.cta_sums[c];
    all += v;
    if (c < (int)blockIdx.x) pre += v;
  }
  pre = block_sum(pre, tmp);
  all = block_sum(all, tmp);
  const unsigned long long kLow = (1ull << 31) - 1;
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    ix.row_ptr[n_keys] = (int)(all >> 31);
    ix.hdr[kHdrNnz] = (int)(all >> 31);
    ix.hdr[kHdrActive] = (int)(all & kLow);
  }
  int lo, hi;
  key_chunk(n_keys, &lo, &hi);
  unsigned long long carry = pre;
  for (int t0 = lo; t0 < hi; t0 += kScanTile) {
    const int k0 = t0 + threadIdx.x * kScanPerThread;
    int c[kScanPerThread];
    unsigned long long local = 0;
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) {
      c[j] = (k0 + j < hi) ? ix.counts[k0 + j] : 0;
      local += key_payload(c[j]);
    }
    if (threadIdx.x == 0) n_long = 0;
    unsigned long long tot;
    unsigned long long run = carry + block_exclusive_scan(local, tmp, &tot);
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) {
      const int key = k0 + j;
      if (key < hi) {
        const int base = (int)(run >> 31);
        ix.row_ptr[key] = base;
        if (c[j] > 0) {
          const int pos = (int)(run & kLow);
          ix.active[pos] = key;
          const int g = key / NB, r = key - g * NB;
          const SeqInfo si = ix.seq[seq_of_block(ix.seq, B, r)];
          const int b = r - si.blk_off;
          const int valid = si.L - 128 * b;
          ix.active_valid[pos] = valid < 128 ? valid : 128;
          if (si.words <= 2) {
            emit_row_serial(ix, ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words, si.words,
                            ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq, si.q_begin, g, Hkv,
                            topk, base);
          } else {
            const int at = atomicAdd(&n_long, 1);
            long_key[at] = key;
            long_base[at] = base;
          }
        }
      }
      run += key_payload(c[j]);
    }
    __syncthreads();
    for (int i = warp; i < n_long; i += n_warps) {
      const int key = long_key[i];
      const int g = key / NB, r = key - g * NB;
      const SeqInfo si = ix.seq[seq_of_block(ix.seq, B, r)];
      const int b = r - si.blk_off;
      emit_row_warp(ix, ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words, si.words,
                    ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq, si.q_begin, g, Hkv, topk,
                    long_base[i]);
    }
    (void)lane;
    __syncthreads();
    carry += tot;
  }
}


constexpr int kIndexThreads = 256;
static_assert(kIndexThreads == kScanThreads && kIndexThreads == kMarkWarps * 32, "phase block sizes");

struct IndexArgs {
  IndexPtrs ix;
  const int32_t* sel;
  const int64_t* cu;
  const int32_t* lens;
  int B, total_q, Hkv, topk, cap_len, causal;
};

// All five index phases with their grid barriers (blockDim.x = kIndexThreads,
// cooperative launch).  `tmp` and `rowbuf` are shared-memory scratch.
__device__ __forceinline__ void build_index_phases(const IndexArgs& a, unsigned long long* tmp,
                                                   int32_t (*rowbuf)[256]) {
  int* bar = a.ix.hdr + kHdrBarCount;
  int epoch = 0;
  int* flags = a.ix.hdr + kHdrFlags;
  const unsigned nb = gridDim.x;
  if (blockIdx.x == 0)
    phase_seq(a.ix, a.cu, a.lens, a.B, a.total_q, a.Hkv, a.cap_len, a.causal, reinterpret_cast<long long*>(tmp));
  phase_token_seq(a.ix, a.cu, a.B, a.total_q);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  phase_zero(a.ix, a.Hkv, SeqTotals{a.ix.hdr[kHdrNB], a.ix.hdr[kHdrBMW], a.ix.hdr[kHdrKMW]});
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  phase_mark(a.ix, a.sel, a.total_q, a.Hkv, a.topk, a.causal, rowbuf);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  phase_key_reduce(a.ix, tmp);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  phase_key_scan_emit(a.ix, a.B, a.Hkv, a.topk, tmp);
}

}  // namespace ixp
}  // namespace mxsa
