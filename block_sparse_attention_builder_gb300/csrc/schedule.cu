// Load-balancing scheduler ("load-balancing scheduler" in the test list of
// the fw-ai/minimax-kernels README; the split rule and the cost model are
// this library's).
//
// Each key with cnt entries becomes n = ceil(cnt / E) work items, item i
// covering entries [i*cnt/n, (i+1)*cnt/n) of the key (E = MXSA_ITEM_TILES
// tiles of 128 (token, head) rows).  An item's integer cost is
//   valid_tokens * kv_weight + tiles * 256 + rows * 2,
// kv_weight = 2 for 16-bit caches and 1 for FP8, modelling the KV bytes
// loaded once per item plus the per-tile tensor/softmax work.  The items
// are laid out in key order and cut into num_ctas contiguous ranges at the
// cost targets floor(c * C / num_ctas): CTA c takes the items whose
// exclusive cost prefix lies in [target_c, target_{c+1}), so no CTA exceeds
// C / num_ctas by more than one item.
//
//   k_sched_init   clears the look-back state
//   k_sched_scan   look-back scan over active keys: item and cost prefixes,
//                  then writes items[] and cost_prefix[]
//   k_partition    one thread per CTA boundary: binary search of the target
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
  int key, begin, cnt, n_items;
  long long cost;
};

__device__ __forceinline__ long long item_cost(int ne, int valid, int kvw, int per_tile, int G) {
  return (long long)valid * kvw + (long long)((ne + per_tile - 1) / per_tile) * 256 + (long long)ne * G * 2;
}

__global__ void k_sched_init(SchedPtrs sc, long long tiles_cap, int num_ctas) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < tiles_cap; i += stride)
    sc.lookback[i] = 0ull;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc.hdr[kSchItems] = 0;
    sc.hdr[kSchCtas] = num_ctas;
    sc.hdr[kSchCostLo] = 0;
    sc.hdr[kSchCostHi] = 0;
    sc.hdr[kSchTileCtr] = 0;
    sc.cost_prefix[0] = 0;
  }
}

__global__ void __launch_bounds__(kScanThreads) k_sched_scan(IndexPtrs ix, SchedPtrs sc, int G, int kvw,
                                                              int per_tile, int E) {
  __shared__ int tile_s;
  __shared__ unsigned long long tmp[33];
  __shared__ unsigned long long excl_s;
  const int n_active = ix.hdr[kHdrActive];
  const int n_tiles = (n_active + kScanTile - 1) / kScanTile;
  if (threadIdx.x == 0) tile_s = atomicAdd(&sc.hdr[kSchTileCtr], 1);
  __syncthreads();
  const int tile = tile_s;
  if (tile >= n_tiles) return;
  const int a0 = tile * kScanTile + threadIdx.x * kScanPerThread;
  KeyWork kw[kScanPerThread];
  unsigned long long local = 0;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    const int a = a0 + j;
    kw[j] = KeyWork{0, 0, 0, 0, 0};
    if (a < n_active) {
      const int key = ix.active[a];
      const int b0 = ix.row_ptr[key], b1 = ix.row_ptr[key + 1];
      const int cnt = b1 - b0;
      const int n = (cnt + E - 1) / E;
      const int valid = ix.active_valid[a];
      long long cost = 0;
      for (int i = 0; i < n; ++i) {
        const int ne = (int)(((long long)(i + 1) * cnt) / n - ((long long)i * cnt) / n);
        cost += item_cost(ne, valid, kvw, per_tile, G);
      }
      kw[j] = KeyWork{key, b0, cnt, n, cost};
      local += ((unsigned long long)cost << kItemBits) | (unsigned long long)n;
    }
  }
  unsigned long long tot;
  unsigned long long ex = block_excl_u64(local, tmp, &tot);
  if (threadIdx.x == 0) excl_s = lookback_exclusive(sc.lookback, tile, tot, &ix.hdr[kHdrFlags]);
  __syncthreads();
  unsigned long long run = excl_s + ex;
  const unsigned long long kLow = (1ull << kItemBits) - 1;
#pragma unroll
  for (int j = 0; j < kScanPerThread; ++j) {
    if (a0 + j >= n_active) break;
    const int valid = ix.active_valid[a0 + j];
    long long item = (long long)(run & kLow);
    long long cost = (long long)(run >> kItemBits);
    const int n = kw[j].n_items, cnt = kw[j].cnt;
    for (int i = 0; i < n; ++i) {
      const int e0 = (int)(((long long)i * cnt) / n), e1 = (int)(((long long)(i + 1) * cnt) / n);
      sc.items[item] = make_int4(kw[j].key, kw[j].begin + e0, e1 - e0, 0);
      sc.cost_prefix[item] = cost;
      cost += item_cost(e1 - e0, valid, kvw, per_tile, G);
      ++item;
    }
    run += ((unsigned long long)kw[j].cost << kItemBits) | (unsigned long long)n;
  }
  if (tile == n_tiles - 1 && threadIdx.x == kScanThreads - 1) {
    const unsigned long long all = excl_s + tot;
    const long long n_items = (long long)(all & kLow);
    const long long C = (long long)(all >> kItemBits);
    sc.hdr[kSchItems] = (int)n_items;
    sc.hdr[kSchCostLo] = (int)(C & 0xffffffffll);
    sc.hdr[kSchCostHi] = (int)(C >> 32);
    sc.cost_prefix[n_items] = C;
  }
}

__global__ void k_partition(SchedPtrs sc, int num_ctas) {
  const int n_items = sc.hdr[kSchItems];
  const long long C = (long long)(unsigned)sc.hdr[kSchCostLo] | ((long long)sc.hdr[kSchCostHi] << 32);
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c <= num_ctas; c += gridDim.x * blockDim.x) {
    const long long target = (long long)c * C / num_ctas;
    // number of items with cost_prefix < target (prefix is non-decreasing)
    int lo = 0, hi = n_items;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sc.cost_prefix[mid] < target) lo = mid + 1;
      else hi = mid;
    }
    sc.cta_ptr[c] = lo;
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
  k_sched_init<<<(int)std::min<long long>((tiles + 255) / 256, 1024), 256, 0, st>>>(sc, tiles, num_ctas);
  if (lay.tiles_cap > 0)
    k_sched_scan<<<(unsigned)lay.tiles_cap, kScanThreads, 0, st>>>(ix, sc, G, kvw, per_tile, E);
  k_partition<<<(num_ctas + 1 + 255) / 256, 256, 0, st>>>(sc, num_ctas);
  return cudaGetLastError();
}

}  // namespace mxsa
