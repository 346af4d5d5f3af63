// Schedule definitions shared by the schedule kernel and the fused plan
// kernel: the per-key and per-item closed forms of the load-balancing
// schedule (see schedule.cu for the rule).
#pragma once
#include "internal.h"

namespace mxsa {
namespace sch {

constexpr int kItemBits = 26;  // payload: (cost << 26) | items
constexpr int kSchThreads = 256;
constexpr int kSchPerThread = 1;
constexpr int kSchTile = kSchThreads * kSchPerThread;

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

// Exclusive scan of three u64 values at once across the CTA (one pass of
// shuffles and one shared-memory exchange for all three).
struct U3 {
  unsigned long long x, y, z;
};

__device__ __forceinline__ U3 block_excl_u64x3(U3 v, unsigned long long* tmp3 /* [3 * 33] */, U3* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  U3 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long a = __shfl_up_sync(0xffffffffu, inc.x, o);
    const unsigned long long b = __shfl_up_sync(0xffffffffu, inc.y, o);
    const unsigned long long c = __shfl_up_sync(0xffffffffu, inc.z, o);
    if (lane >= o) {
      inc.x += a;
      inc.y += b;
      inc.z += c;
    }
  }
  if (lane == 31) {
    tmp3[warp] = inc.x;
    tmp3[33 + warp] = inc.y;
    tmp3[66 + warp] = inc.z;
  }
  __syncthreads();
  if (warp < 3) {
    unsigned long long* t = tmp3 + 33 * warp;
    const unsigned long long w = lane < nw ? t[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long a = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += a;
    }
    if (lane < nw) t[lane] = wi - w;
    if (lane == nw - 1) t[32] = wi;
  }
  __syncthreads();
  U3 r{tmp3[warp] + inc.x - v.x, tmp3[33 + warp] + inc.y - v.y, tmp3[66 + warp] + inc.z - v.z};
  *total = U3{tmp3[32], tmp3[65], tmp3[98]};
  __syncthreads();
  return r;
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

struct Params {
  int B, Hkv, G, kvw, per_tile, E, num_ctas, topk;
};

// What one active key contributes.  kind 0: nothing (inside a decode run),
// 1: a normal key, 2: the first key of a decode run.
struct KeyWork {
  int kind;
  int a;      // active position
  int key;    // normal: key id
  int begin;  // normal: first entry
  int cnt;    // normal: entries; decode: run length (keys)
  int valid;  // normal: valid tokens of the block
  int adj;    // decode: cost removed from the run's last item (partial last block)
  int n;      // items
  long long cost;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// exclusive cost prefix of item i within a normal key, and item i's cost
// Cost units where a 128-row tile costs 256: a normal item's fixed part
// (its stage turnover: the block's load, and for FP8 its widening, before
// its first tile) and the per-row part (gather, epilogue stores).  Chosen by
// timing a mixed FP8 varlen batch over a sweep of both constants.
constexpr long long kItemFixed = 384;
constexpr long long kRowCost = 3;

__device__ __forceinline__ void normal_item(const KeyWork& k, const Params& P, int i, int* e0, int* ne,
                                            long long* pre, long long* cost) {
  const int q = k.cnt / k.n;
  const long long fl = (long long)i * k.cnt / k.n, fl1 = (long long)(i + 1) * k.cnt / k.n;
  const long long m = fl - (long long)i * q;  // items before i with q + 1 entries
  const long long t_q = ceil_div(q, P.per_tile), t_q1 = ceil_div(q + 1, P.per_tile);
  *e0 = (int)fl;
  *ne = (int)(fl1 - fl);
  *pre = (long long)i * (kItemFixed + (long long)k.valid * P.kvw) + ((i - m) * t_q + m * t_q1) * 256 +
         fl * P.G * kRowCost;
  *cost = kItemFixed + (long long)k.valid * P.kvw + (long long)ceil_div(*ne, P.per_tile) * 256 +
          (long long)(*ne) * P.G * kRowCost;
}

__device__ __forceinline__ void decode_item(const KeyWork& k, const Params& P, int i, int* k0, int* nk,
                                            long long* pre, long long* cost) {
  const long long per_key = 64 + 128LL * P.kvw;
  const int a0 = (int)((long long)i * k.cnt / k.n), a1 = (int)((long long)(i + 1) * k.cnt / k.n);
  *k0 = a0;
  *nk = a1 - a0;
  *pre = (long long)a0 * per_key + (long long)i * 256;
  *cost = (long long)(a1 - a0) * per_key + 256 - (i == k.n - 1 ? k.adj : 0);
}

__device__ __forceinline__ unsigned long long pack(long long cost, int n) {
  return ((unsigned long long)cost << kItemBits) | (unsigned long long)n;
}

__device__ __forceinline__ void active_chunk(int n_active, int* lo, int* hi) {
  const long long chunk = ((long long)n_active + gridDim.x - 1) / gridDim.x;
  const long long a = (long long)blockIdx.x * chunk, b = a + chunk;
  *lo = (int)(a < n_active ? a : n_active);
  *hi = (int)(b < n_active ? b : n_active);
}

// number of boundaries c in [0, P] whose target floor(c * C / P) is <= x
__device__ __forceinline__ int boundaries_at_or_below(long long x, long long C, int P) {
  if (C <= 0) return P + 1;
  const long long n = ((x + 1) * P - 1) / C + 1;
  return (int)(n < P + 1 ? n : P + 1);
}


}  // namespace sch
}  // namespace mxsa
