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
  __shared__ int cu_bad;
  long long carry_blk = 0, carry_bm = 0, carry_km = 0;
  int flags = 0;
  // cu_seqlens_q must be a non-decreasing partition of [0, total_q]; if it is
  // not, every sequence is treated as having no new tokens (nothing indexed),
  // which keeps all per-sequence regions inside their shape-derived bounds
  if (threadIdx.x == 0) cu_bad = (cu[0] != 0 || cu[B] != (int64_t)total_q) ? 1 : 0;
  __syncthreads();
  for (int s = threadIdx.x; s < B; s += blockDim.x)
    if (cu[s + 1] < cu[s]) cu_bad = 1;
  __syncthreads();
  const bool cu_ok = cu_bad == 0;
  if (!cu_ok) flags |= MXSA_FLAG_CU;
  for (int base = 0; base < B; base += blockDim.x) {
    const int s = base + threadIdx.x;
    long long nblk = 0, bmw = 0, kmw = 0;
    int L = 0, tq = 0, q0 = 0, words = 0;
    if (s < B) {
      const int64_t c0 = cu[s], c1 = cu[s + 1];
      tq = cu_ok ? (int)(c1 - c0) : 0;
      q0 = cu_ok ? (int)c0 : 0;
      int Lr = lens[s];
      if (Lr < 0 || Lr > cap_len) flags |= MXSA_FLAG_LEN;
      L = Lr < 0 ? 0 : (Lr > cap_len ? cap_len : Lr);
      if (causal && L < tq) flags |= MXSA_FLAG_CAUSAL_LEN;
      nblk = (L + 127) / 128;
      words = (tq + 31) / 32;
      bmw = nblk * words;
      kmw = nblk * tq;
    }
    long long tb, tbm, tkm;
    long long eb = block_exclusive_scan(nblk, tmp, &tb);
    long long ebm = block_exclusive_scan(bmw, tmp, &tbm);
    long long ekm = block_exclusive_scan(kmw, tmp, &tkm);
    if (tab != nullptr && s < B && B <= kSeqTab) {
      tab[0][s] = (int)(carry_blk + eb);
      tab[1][s] = (int)(carry_bm + ebm);
      tab[2][s] = (int)(carry_km + ekm);
      tab[3][s] = q0;
      tab[4][s] = L;
      tab[5][s] = tq;
    }
    if (s < B && writer) {
      SeqInfo si;
      si.L = L;
      si.nblk = (int)nblk;
      si.blk_off = (int)(carry_blk + eb);
      si.tq = tq;
      si.q_begin = q0;
      si.bm_off = (int)(carry_bm + ebm);
      si.km_off = (int)(carry_km + ekm);
      si.words = words;
      ix.seq[s] = si;
    }
    carry_blk += tb;
    carry_bm += tbm;
    carry_km += tkm;
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

__device__ __forceinline__ void phase_token_seq(const IndexPtrs& ix, const int64_t* cu, int B, int total_q) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long t = tid; t < total_q; t += stride) {
    // last s with cu[s] <= t (sequences of zero tokens are skipped naturally)
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    ix.token_seq[t] = lo;
  }
}

constexpr int kMarkWarps = 8;

// count = false leaves counts alone (the caller derives them from the
// bitmap rows), so popular blocks cost no contended atomics.
__device__ __forceinline__ void phase_mark(const IndexPtrs& ix, const int32_t* sel, int total_q, int Hkv, int topk, int causal,
                           int32_t (*rowbuf)[256], bool count = true) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const long long n_rows = (long long)total_q * Hkv;
  int flags = 0, made = 0, bmin = 0x7fffffff, bmax = -1;
  for (long long row = (long long)blockIdx.x * kMarkWarps + w; row < n_rows; row += (long long)gridDim.x * kMarkWarps) {
    const int t = (int)(row / Hkv), g = (int)(row % Hkv);
    const int32_t* srow = sel + row * topk;
    for (int k = lane; k < topk; k += 32) rowbuf[w][k] = srow[k];
    __syncwarp();
    const int s = ix.token_seq[t];
    const SeqInfo si = ix.seq[s];
    const int i = t - si.q_begin;
    const bool in_seq = i >= 0 && i < si.tq;
    const int pos = si.L - si.tq + i;
    for (int k = lane; k < topk; k += 32) {
      const long long slot = row * topk + k;
      ix.slot_entry[slot] = -1;
      const int b = rowbuf[w][k];
      if (b == -1 || !in_seq) continue;
      if (b < -1 || b >= si.nblk) {
        flags |= MXSA_FLAG_SEL_RANGE;
        continue;
      }
      bool dup = false;
      for (int k2 = 0; k2 < k; ++k2) dup |= rowbuf[w][k2] == b;
      if (dup) {
        flags |= MXSA_FLAG_SEL_DUP;
        continue;
      }
      if (causal && 128 * b > pos) continue;  // block entirely after the token
      const size_t word = (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words + (i >> 5);
      atomicOr(&ix.bitmap[word], 1u << (i & 31));
      ix.kmap[(size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq + i] = (uint8_t)k;
      if (count) atomicAdd(&ix.counts[(long long)g * NB + si.blk_off + b], 1);
      ++made;
      bmin = min(bmin, b);
      bmax = max(bmax, b);
    }
    made = __reduce_add_sync(0xffffffffu, made);
    bmin = __reduce_min_sync(0xffffffffu, bmin);
    bmax = __reduce_max_sync(0xffffffffu, bmax);
    if (lane == 0) {
      ix.row_nnz[row] = made;
      ix.row_minb[row] = bmin;
      ix.row_maxb[row] = bmax;
    }
    made = 0;
    bmin = 0x7fffffff;
    bmax = -1;
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

// Writes the entries of one bitmap row: `n_words` words starting at `bm`,
// for tokens q_begin + 32 w + bit.  Serial over the row (one lane).
__device__ __forceinline__ void emit_row_serial(const IndexPtrs& ix, const uint32_t* bm, int n_words,
                                                const uint8_t* km, int q_begin, int g, int Hkv, int topk,
                                                int base) {
  int j = base;
  for (int w = 0; w < n_words; ++w) {
    uint32_t bits = bm[w];
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      const int i = w * 32 + bit;
      const int k = km[i];
      const int slot = ((q_begin + i) * Hkv + g) * topk + k;
      ix.entries[j] = slot;
      ix.slot_entry[slot] = j;
      ++j;
    }
  }
}

// One warp writes the entries of a long bitmap row, 32 words at a time
// with a prefix over the words' popcounts.
__device__ __forceinline__ void emit_row_warp(const IndexPtrs& ix, const uint32_t* bm, int n_words,
                                              const uint8_t* km, int q_begin, int g, int Hkv, int topk, int base) {
  const int lane = threadIdx.x & 31;
  int run = base;
  for (int w0 = 0; w0 < n_words; w0 += 32) {
    const int w = w0 + lane;
    uint32_t bits = w < n_words ? bm[w] : 0u;
    const int cnt = __popc(bits);
    const int inc = warp_inclusive_scan(cnt);
    int j = run + inc - cnt;
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      const int i = w * 32 + bit;
      const int k = km[i];
      const int slot = ((q_begin + i) * Hkv + g) * topk + k;
      ix.entries[j] = slot;
      ix.slot_entry[slot] = j;
      ++j;
    }
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
    uint32_t bits = w < n_words ? bm[w] : 0u;
    const int cnt = __popc(bits);
    const int inc = warp_inclusive_scan(cnt);
    int j = run + inc - cnt;
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      const int i = w * 32 + bit;
      const int k = km[i];
      const int slot = ((q_begin + i) * Hkv + g) * topk + k;
      ix.entries[j] = slot;
      ix.slot_entry[slot] = j;
      ++j;
    }
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
