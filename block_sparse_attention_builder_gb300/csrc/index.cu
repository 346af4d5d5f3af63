// Index builder: inverts the query -> block selections into block -> entry
// lists ("index builder" in the test list of the fw-ai/minimax-kernels
// README; the algorithm is this library's).
//
// Keys are (kv head g, sequence s, block b) -> key = g * NB + blk_off[s] + b.
// Within a key the entries are the selection slots (t * Hkv + g) * topk + k
// in increasing token order.  The result is deterministic because the order
// never depends on atomics: each (key, token) pair owns one bit of a per-key
// token bitmap, and the emission walks the set bits in order.
//
//   k_seq    (1 CTA)  per-sequence scan: L, nblk, block / bitmap / kmap offsets
//   k_zero   (grid)   clears counters, bitmap and scan state; token -> sequence
//   k_mark   (grid)   one warp per (token, kv head) row: validate, dedupe,
//                     set the token's bit in each selected key row, record k
//   k_scan   (grid)   decoupled look-back scan of per-key counts: row_ptr and
//                     the compacted list of keys with entries
//   k_emit   (grid)   each active key enumerates its bitmap row in order and
//                     writes entries[] and the inverse map slot_entry[]
#include "internal.h"

namespace mxsa {

namespace {

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

__global__ void __launch_bounds__(1024) k_seq(IndexPtrs ix, const int64_t* cu, const int32_t* lens, int B,
                                              int total_q, int Hkv, int cap_len, int causal) {
  __shared__ long long tmp[33];
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
    if (s < B) {
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
  if (threadIdx.x == 0) {
    ix.hdr[kHdrFlags] = fl;
    ix.hdr[kHdrNB] = (int)carry_blk;
    ix.hdr[kHdrNnz] = 0;
    ix.hdr[kHdrActive] = 0;
    ix.hdr[kHdrKeys] = (int)(carry_blk * Hkv);
    ix.hdr[kHdrBMW] = (int)carry_bm;
    ix.hdr[kHdrKMW] = (int)carry_km;
    ix.hdr[kHdrTileCtr] = 0;
    ix.row_ptr[0] = 0;
  }
}

__global__ void k_zero(IndexPtrs ix, const int64_t* cu, int B, int total_q, int Hkv) {
  const long long n_keys = ix.hdr[kHdrKeys];
  const long long n_bm = (long long)ix.hdr[kHdrBMW] * Hkv;
  const long long n_tiles = (n_keys + kScanTile - 1) / kScanTile;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long i = tid; i < n_keys; i += stride) ix.counts[i] = 0;
  for (long long i = tid; i < n_bm; i += stride) ix.bitmap[i] = 0u;
  for (long long i = tid; i < n_tiles; i += stride) ix.lookback[i] = 0ull;
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

__global__ void __launch_bounds__(kMarkWarps * 32) k_mark(IndexPtrs ix, const int32_t* sel, int total_q, int Hkv,
                                                         int topk, int causal) {
  __shared__ int32_t rowbuf[kMarkWarps][256];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const long long n_rows = (long long)total_q * Hkv;
  int flags = 0;
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
      atomicAdd(&ix.counts[(long long)g * NB + si.blk_off + b], 1);
    }
    __syncwarp();
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(&ix.hdr[kHdrFlags], flags);
}

// Look-back scan over keys; payload = (entry count << 31) | active count.
__global__ void __launch_bounds__(kScanThreads) k_scan(IndexPtrs ix) {
  __shared__ int tile_s;
  __shared__ unsigned long long tmp[33];
  __shared__ unsigned long long excl_s;
  const int n_keys = ix.hdr[kHdrKeys];
  const int n_tiles = (n_keys + kScanTile - 1) / kScanTile;
  if (threadIdx.x == 0) tile_s = atomicAdd(&ix.hdr[kHdrTileCtr], 1);
  __syncthreads();
  const int tile = tile_s;
  if (tile >= n_tiles) return;
  const long long k0 = (long long)tile * kScanTile + threadIdx.x * kScanPerThread;
  int c[kScanPerThread];
  unsigned long long local = 0;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    c[j] = (k0 + j < n_keys) ? ix.counts[k0 + j] : 0;
    local += ((unsigned long long)c[j] << 31) | (c[j] > 0 ? 1ull : 0ull);
  }
  unsigned long long tot;
  unsigned long long ex = block_exclusive_scan(local, tmp, &tot);
  if (threadIdx.x == 0) excl_s = lookback_exclusive(ix.lookback, tile, tot, &ix.hdr[kHdrFlags]);
  __syncthreads();
  unsigned long long run = excl_s + ex;
  const unsigned long long kLow = (1ull << 31) - 1;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    if (k0 + j < n_keys) {
      ix.row_ptr[k0 + j] = (int)(run >> 31);
      if (c[j] > 0) ix.active[run & kLow] = (int)(k0 + j);
    }
    run += ((unsigned long long)c[j] << 31) | (c[j] > 0 ? 1ull : 0ull);
  }
  if (tile == n_tiles - 1 && threadIdx.x == kScanThreads - 1) {
    const unsigned long long all = excl_s + tot;
    ix.row_ptr[n_keys] = (int)(all >> 31);
    ix.hdr[kHdrNnz] = (int)(all >> 31);
    ix.hdr[kHdrActive] = (int)(all & kLow);
  }
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

__global__ void __launch_bounds__(256) k_emit(IndexPtrs ix, int B, int Hkv, int topk) {
  const int lane = threadIdx.x & 31;
  const int n_active = ix.hdr[kHdrActive];
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int grp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); grp * 32 < n_active; grp += warps_total) {
    const int a = grp * 32 + lane;
    bool have = a < n_active;
    int key = 0, g = 0, s = 0, b = 0, words = 0, base = 0;
    SeqInfo si{};
    if (have) {
      key = ix.active[a];
      g = key / NB;
      const int r = key - g * NB;
      s = seq_of_block(ix.seq, B, r);
      si = ix.seq[s];
      b = r - si.blk_off;
      words = si.words;
      base = ix.row_ptr[key];
      const int valid = si.L - 128 * b;
      ix.active_valid[a] = valid < 128 ? valid : 128;
    }
    const uint32_t* bm = ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * words;
    const uint8_t* km = ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq;
    // short rows (<= 2 words): one lane per key
    const bool is_long = have && words > 2;
    if (have && !is_long) emit_row_serial(ix, bm, words, km, si.q_begin, g, Hkv, topk, base);
    // long rows: the warp walks 32 words at a time with a prefix over popcounts
    unsigned long_mask = __ballot_sync(0xffffffffu, is_long);
    while (long_mask) {
      const int src = __ffs(long_mask) - 1;
      long_mask &= long_mask - 1;
      const int L_words = __shfl_sync(0xffffffffu, words, src);
      const int L_base = __shfl_sync(0xffffffffu, base, src);
      const int L_g = __shfl_sync(0xffffffffu, g, src);
      const int L_q0 = __shfl_sync(0xffffffffu, si.q_begin, src);
      const unsigned long long bm_addr = __shfl_sync(0xffffffffu, (unsigned long long)bm, src);
      const unsigned long long km_addr = __shfl_sync(0xffffffffu, (unsigned long long)km, src);
      const uint32_t* lbm = reinterpret_cast<const uint32_t*>(bm_addr);
      const uint8_t* lkm = reinterpret_cast<const uint8_t*>(km_addr);
      int run = L_base;
      for (int w0 = 0; w0 < L_words; w0 += 32) {
        const int w = w0 + lane;
        uint32_t bits = w < L_words ? lbm[w] : 0u;
        const int cnt = __popc(bits);
        const int inc = warp_inclusive_scan(cnt);
        int j = run + inc - cnt;
        while (bits) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          const int i = w * 32 + bit;
          const int k = lkm[i];
          const int slot = ((L_q0 + i) * Hkv + L_g) * topk + k;
          ix.entries[j] = slot;
          ix.slot_entry[slot] = j;
          ++j;
        }
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
  }
}

}  // namespace

cudaError_t launch_build_index(const mxsa_problem& p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                               const IndexPtrs& ix, const mxsa_index_layout& lay, cudaStream_t st) {
  const int cap_len = p.max_pages_per_seq * p.page_size;
  k_seq<<<1, 1024, 0, st>>>(ix, cu, lens, p.num_seqs, p.total_q, p.num_kv_heads, cap_len, p.causal);
  int sms = 148;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  k_zero<<<sms * 4, 256, 0, st>>>(ix, cu, p.num_seqs, p.total_q, p.num_kv_heads);
  const long long rows = (long long)p.total_q * p.num_kv_heads;
  if (rows > 0) {
    long long g = (rows + kMarkWarps - 1) / kMarkWarps;
    if (g > sms * 16) g = sms * 16;
    k_mark<<<(int)g, kMarkWarps * 32, 0, st>>>(ix, sel, p.total_q, p.num_kv_heads, p.topk, p.causal);
  }
  if (lay.tiles_cap > 0) k_scan<<<(unsigned)lay.tiles_cap, kScanThreads, 0, st>>>(ix);
  long long groups = (std::min<long long>(lay.keys_cap, lay.nslots) + 31) / 32;
  long long eg = (groups + 7) / 8;
  if (eg > sms * 8) eg = sms * 8;
  if (eg < 1) eg = 1;
  k_emit<<<(int)eg, 256, 0, st>>>(ix, p.num_seqs, p.num_kv_heads, p.topk);
  return cudaGetLastError();
}

}  // namespace mxsa
