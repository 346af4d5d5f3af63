// Load-balancing scheduler ("load-balancing scheduler" in the test list of
// the fw-ai/minimax-kernels README; the split rule, the decode merge and the
// cost model are this library's).
//
// Active keys (keys with entries) are taken in key order and produce two
// work lists:
//  * normal keys (sequences with several new tokens): n = ceil(cnt / E)
//    items of <= E = MXSA_ITEM_TILES * (128 / G) entries, item i covering
//    entries [i*cnt/n, (i+1)*cnt/n) of the key; cost =
//    valid_tokens * kv_weight + tiles * 256 + rows * 2;
//  * decode keys (sequences with one new token, G <= 16): every key of one
//    (kv head, sequence) holds the same single entry, so the run of such
//    keys is cut into ceil(len / 8) items of consecutive keys that the
//    decode forward processes with one online softmax; cost =
//    sum(valid_tokens * kv_weight) + keys * 64 + 256.
// kv_weight = 2 for 16-bit caches and 1 for FP8.  Each list is laid out in
// key order and cut into num_ctas contiguous ranges at the cost targets
// floor(c * C / num_ctas): CTA c takes the items whose exclusive cost prefix
// lies in [target_c, target_{c+1}), so no CTA exceeds C / num_ctas by more
// than one item.
//
//   k_sched_init   clears the look-back state
//   k_sched_scan   look-back scans over active keys (one per list), then
//                  writes the items and their cost prefixes
//   k_partition    one thread per CTA boundary and list: binary search
#include <algorithm>

#include "internal.h"

namespace mxsa {

namespace {

constexpr int kItemBits = 26;  // payload: (cost << 26) | items

__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__device__ __forceinline__ unsigned long long block_excl_u64(unsigned long long v, unsigned long long* tmp,
                                                             unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned long long inc = warp_incl_u64(v);
  if (lane == 31) tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < nw ? tmp[lane] : 0ull;
    unsigned long long wi = warp_incl_u64(w);
    if (lane < nw) tmp[lane] = wi - w;
    if (lane == nw - 1) tmp[32] = wi;
  }
  __syncthreads();
  unsigned long long r = tmp[warp] + inc - v;
  *total = tmp[32];
  __syncthreads();
  return r;
}

struct KeyWork {
  int key, begin, cnt, n_items;  // normal key; n_items = 0 when not emitting
  long long cost;
  int dec_len, dec_items;        // decode run start: run length and items
  long long dec_cost;
};

__device__ __forceinline__ long long item_cost(int ne, int valid, int kvw, int per_tile, int G) {
  return (long long)valid * kvw + (long long)((ne + per_tile - 1) / per_tile) * 256 + (long long)ne * G * 2;
}

__device__ __forceinline__ int seq_of_block(const SeqInfo* seq, int B, int r) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq[mid].blk_off <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// decode run of `len` keys starting at active position a: cost of its
// chunk [k0, k1)
__device__ __forceinline__ long long dec_chunk_cost(const IndexPtrs& ix, int a, int k0, int k1, int kvw) {
  long long c = (long long)(k1 - k0) * 64 + 256;
  for (int k = k0; k < k1; ++k) c += (long long)ix.active_valid[a + k] * kvw;
  return c;
}

__global__ void k_sched_init(SchedPtrs sc, long long tiles_cap, int num_ctas) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * tiles_cap; i += stride)
    sc.lookback[i] = 0ull;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc.hdr[kSchItems] = 0;
    sc.hdr[kSchCtas] = num_ctas;
    sc.hdr[kSchCostLo] = 0;
    sc.hdr[kSchCostHi] = 0;
    sc.hdr[kSchTileCtr] = 0;
    sc.hdr[kSchDecItems] = 0;
    sc.hdr[kSchDecCostLo] = 0;
    sc.hdr[kSchDecCostHi] = 0;
    sc.cost_prefix[0] = 0;
    sc.cost_prefix_dec[0] = 0;
  }
}

__global__ void __launch_bounds__(kScanThreads) k_sched_scan(IndexPtrs ix, SchedPtrs sc, long long tiles_cap,
                                                              int B, int G, int kvw, int per_tile, int E) {
  __shared__ int tile_s;
  __shared__ unsigned long long tmp[33];
  __shared__ unsigned long long excl_n, excl_d;
  const int n_active = ix.hdr[kHdrActive];
  const int NB = ix.hdr[kHdrNB];
  const int n_tiles = (n_active + kScanTile - 1) / kScanTile;
  if (threadIdx.x == 0) tile_s = atomicAdd(&sc.hdr[kSchTileCtr], 1);
  __syncthreads();
  const int tile = tile_s;
  if (tile >= n_tiles) return;
  const bool dec_ok = G <= kDecodeMaxG;
  const int a0 = tile * kScanTile + threadIdx.x * kScanPerThread;
  KeyWork kw[kScanPerThread];
  unsigned long long local_n = 0, local_d = 0;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    const int a = a0 + j;
    kw[j] = KeyWork{0, 0, 0, 0, 0, 0, 0, 0};
    if (a >= n_active) continue;
    const int key = ix.active[a];
    const int g = key / NB, r = key - g * NB;
    const SeqInfo si = ix.seq[seq_of_block(ix.seq, B, r)];
    if (!(dec_ok && si.tq == 1)) {
      const int b0 = ix.row_ptr[key], b1 = ix.row_ptr[key + 1];
      const int cnt = b1 - b0;
      const int n = (cnt + E - 1) / E;
      const int valid = ix.active_valid[a];
      long long cost = 0;
      for (int i = 0; i < n; ++i) {
        const int ne = (int)(((long long)(i + 1) * cnt) / n - ((long long)i * cnt) / n);
        cost += item_cost(ne, valid, kvw, per_tile, G);
      }
      kw[j].key = key;
      kw[j].begin = b0;
      kw[j].cnt = cnt;
      kw[j].n_items = n;
      kw[j].cost = cost;
      local_n += ((unsigned long long)cost << kItemBits) | (unsigned long long)n;
    } else {
      const int lo = g * NB + si.blk_off, hi = lo + si.nblk;  // keys of this (g, s)
      if (a > 0 && ix.active[a - 1] >= lo) continue;          // not the first key of its run
      int len = 1;
      while (a + len < n_active && ix.active[a + len] < hi) ++len;
      const int n = (len + kDecodeBlocks - 1) / kDecodeBlocks;
      long long cost = 0;
      for (int i = 0; i < n; ++i) cost += dec_chunk_cost(ix, a, (i * len) / n, ((i + 1) * len) / n, kvw);
      kw[j].dec_len = len;
      kw[j].dec_items = n;
      kw[j].dec_cost = cost;
      local_d += ((unsigned long long)cost << kItemBits) | (unsigned long long)n;
    }
  }
  unsigned long long tot_n, tot_d;
  const unsigned long long ex_n = block_excl_u64(local_n, tmp, &tot_n);
  const unsigned long long ex_d = block_excl_u64(local_d, tmp, &tot_d);
  if (threadIdx.x == 0) {
    excl_n = lookback_exclusive(sc.lookback, tile, tot_n, &ix.hdr[kHdrFlags]);
    excl_d = lookback_exclusive(sc.lookback + tiles_cap, tile, tot_d, &ix.hdr[kHdrFlags]);
  }
  __syncthreads();
  const unsigned long long kLow = (1ull << kItemBits) - 1;
  unsigned long long run_n = excl_n + ex_n, run_d = excl_d + ex_d;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    const int a = a0 + j;
    if (a >= n_active) break;
    if (kw[j].n_items > 0) {
      const int valid = ix.active_valid[a];
      long long item = (long long)(run_n & kLow);
      long long cost = (long long)(run_n >> kItemBits);
      const int n = kw[j].n_items, cnt = kw[j].cnt;
      for (int i = 0; i < n; ++i) {
        const int e0 = (int)(((long long)i * cnt) / n), e1 = (int)(((long long)(i + 1) * cnt) / n);
        sc.items[item] = make_int4(kw[j].key, kw[j].begin + e0, e1 - e0, 0);
        sc.cost_prefix[item] = cost;
        cost += item_cost(e1 - e0, valid, kvw, per_tile, G);
        ++item;
      }
      run_n += ((unsigned long long)kw[j].cost << kItemBits) | (unsigned long long)n;
    }
    if (kw[j].dec_items > 0) {
      long long item = (long long)(run_d & kLow);
      long long cost = (long long)(run_d >> kItemBits);
      const int n = kw[j].dec_items, len = kw[j].dec_len;
      for (int i = 0; i < n; ++i) {
        const int k0 = (i * len) / n, k1 = ((i + 1) * len) / n;
        sc.items_dec[item] = make_int4(a + k0, ix.row_ptr[ix.active[a + k0]], 1, k1 - k0);
        sc.cost_prefix_dec[item] = cost;
        cost += dec_chunk_cost(ix, a, k0, k1, kvw);
        ++item;
      }
      run_d += ((unsigned long long)kw[j].dec_cost << kItemBits) | (unsigned long long)n;
    }
  }
  if (tile == n_tiles - 1 && threadIdx.x == kScanThreads - 1) {
    const unsigned long long all_n = excl_n + tot_n, all_d = excl_d + tot_d;
    const long long nn = (long long)(all_n & kLow), Cn = (long long)(all_n >> kItemBits);
    const long long nd = (long long)(all_d & kLow), Cd = (long long)(all_d >> kItemBits);
    sc.hdr[kSchItems] = (int)nn;
    sc.hdr[kSchCostLo] = (int)(Cn & 0xffffffffll);
    sc.hdr[kSchCostHi] = (int)(Cn >> 32);
    sc.cost_prefix[nn] = Cn;
    sc.hdr[kSchDecItems] = (int)nd;
    sc.hdr[kSchDecCostLo] = (int)(Cd & 0xffffffffll);
    sc.hdr[kSchDecCostHi] = (int)(Cd >> 32);
    sc.cost_prefix_dec[nd] = Cd;
  }
}

__global__ void k_partition(SchedPtrs sc, int num_ctas) {
  for (int c2 = blockIdx.x * blockDim.x + threadIdx.x; c2 < 2 * (num_ctas + 1); c2 += gridDim.x * blockDim.x) {
    const bool dec = c2 > num_ctas;
    const int c = dec ? c2 - (num_ctas + 1) : c2;
    const int n_items = sc.hdr[dec ? kSchDecItems : kSchItems];
    const long long C = (long long)(unsigned)sc.hdr[dec ? kSchDecCostLo : kSchCostLo] |
                        ((long long)sc.hdr[dec ? kSchDecCostHi : kSchCostHi] << 32);
    const long long* prefix = dec ? sc.cost_prefix_dec : sc.cost_prefix;
    const long long target = (long long)c * C / num_ctas;
    // number of items with cost_prefix < target (prefix is non-decreasing)
    int lo = 0, hi = n_items;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] < target) lo = mid + 1;
      else hi = mid;
    }
    (dec ? sc.cta_ptr_dec : sc.cta_ptr)[c] = lo;
  }
}

}  // namespace

cudaError_t launch_schedule(const mxsa_problem& p, const IndexPtrs& ix, const SchedPtrs& sc,
                            const mxsa_sched_layout& lay, int num_ctas, cudaStream_t st) {
  const int G = p.num_q_heads / p.num_kv_heads;
  const int per_tile = std::max(1, MXSA_TILE_ROWS / G);
  const int E = MXSA_ITEM_TILES * per_tile;
  const int kvw = p.kv_dtype == MXSA_FP8_E4M3 ? 1 : 2;
  const long long tiles = std::max<long long>(lay.tiles_cap, 1);
  k_sched_init<<<(int)std::min<long long>((2 * tiles + 255) / 256, 1024), 256, 0, st>>>(sc, tiles, num_ctas);
  if (lay.tiles_cap > 0)
    k_sched_scan<<<(unsigned)lay.tiles_cap, kScanThreads, 0, st>>>(ix, sc, tiles, p.num_seqs, G, kvw, per_tile,
                                                                     E);
  k_partition<<<(2 * (num_ctas + 1) + 255) / 256, 256, 0, st>>>(sc, num_ctas);
  return cudaGetLastError();
}

}  // namespace mxsa
