// Load-balancing scheduler ("load-balancing scheduler" in the test list of
// the fw-ai/minimax-kernels README; the split rule, the decode merge and the
// cost model are this library's).
//
// Active keys (keys with entries) are taken in key order and produce two
// work lists:
//  * decode keys: a key of a sequence with one new token (G <= 16) that
//    holds exactly one entry, of that token.  A maximal run of consecutive
//    active decode keys of one (kv head, sequence) is cut into
//    ceil(len / 8) items of consecutive keys that the decode forward
//    processes with one online softmax; cost =
//    sum(valid_tokens * kv_weight) + keys * 64 + 256.  With the plain index
//    every key of such a sequence is a decode key; with the dedup index a
//    key of a shared block holds several sequences' entries and is a normal
//    key;
//  * normal keys (every other key): n = ceil(cnt / E) items of
//    <= E = MXSA_ITEM_TILES * (128 / G) entries, item i covering entries
//    [i*cnt/n, (i+1)*cnt/n) of the key; cost =
//    valid_tokens * kv_weight + tiles * 256 + rows * 2.
// kv_weight = 2 for 16-bit caches and 1 for FP8.  Each list is laid out in
// key order and cut into num_ctas contiguous ranges at the cost targets
// floor(c * C / num_ctas): CTA c takes the items whose exclusive cost prefix
// lies in [target_c, target_{c+1}), so no CTA exceeds C / num_ctas by more
// than one item.
//
// Every per-key and per-item quantity has a closed form (item sizes take
// two values, q = cnt / n and q + 1, and the first i items hold
// floor(i * cnt / n) entries), so the work per key and per item is O(1);
// a decode run's length is found from a bit per active key (is it a decode
// key) and the run's (kv head, sequence) key range.  One cooperative launch,
// three phases separated by bounded grid barriers (the fused plan kernel in
// plan.cu computes the same schedule of a plain index inside its build):
//   flags   one warp per 32 active keys writes their decode-key bits
//   reduce  the active keys are cut into one contiguous chunk per CTA; each
//           CTA sums the item counts and costs of its chunk (both lists)
//   scan    each CTA adds the sums of the chunks before it, scans its chunk
//           in tiles and writes the tile's items in parallel; an item with
//           exclusive prefix p and cost w sets cta_ptr[c] = item + 1 for
//           every boundary c whose target lies in (p, p + w], which is the
//           partition rule above without a search
#include <algorithm>

#include "index_phases.cuh"
#include "sched_common.cuh"

namespace mxsa {

namespace {

using namespace sch;

__device__ __forceinline__ bool dk_bit(const uint32_t* dk, int a) { return (dk[a >> 5] >> (a & 31)) & 1u; }

// flags: bit a of sc.dk = active key a is a decode key
__device__ void phase_flags(const IndexPtrs& ix, const SchedPtrs& sc, const Params& P) {
  const int n_active = ix.hdr[kHdrActive], NB = ix.hdr[kHdrNB];
  const int lane = threadIdx.x & 31;
  const long long n_words = ((long long)n_active + 31) / 32;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n_words; w += warps) {
    const int a = (int)(w * 32) + lane;
    bool d = false;
    if (a < n_active && P.G <= kDecodeMaxG) {
      const int key = ix.active[a];
      const int g = key / NB, r = key - g * NB;
      const SeqInfo si = ix.seq[seq_of_block(ix.seq, P.B, r)];
      if (si.tq == 1) {
        const int beg = ix.row_ptr[key];
        if (ix.row_ptr[key + 1] - beg == 1) d = ix.entries[beg] / (P.Hkv * P.topk) == si.q_begin;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, d);
    if (lane == 0) sc.dk[w] = m;
  }
}

// first active position in (a, limit) that is not a decode key, or limit
__device__ __forceinline__ int next_non_decode(const uint32_t* dk, int a, int limit) {
  int e = a + 1;
  while (e < limit) {
    const int sh = e & 31;
    const uint32_t inv = ~(dk[e >> 5] >> sh);  // bit j: key e + j is not a decode key (or lies past the word)
    const int z = __ffs(inv) - 1;
    if (z >= 0 && z < 32 - sh) {
      e += z;
      break;
    }
    e += 32 - sh;
  }
  return e < limit ? e : limit;
}

// chunk_end: keys from chunk_end on belong to the next CTA (nothing to do)
__device__ __forceinline__ KeyWork key_work(const IndexPtrs& ix, const SchedPtrs& sc, const Params& P, int NB,
                                            int chunk_end, int n_active, int a) {
  KeyWork w{};
  w.a = a;
  if (a >= chunk_end) return w;
  const int key = ix.active[a];
  if (dk_bit(sc.dk, a)) {
    const int g = key / NB, r = key - g * NB;
    const SeqInfo si = ix.seq[seq_of_block(ix.seq, P.B, r)];
    const int lo = g * NB + si.blk_off, hi = lo + si.nblk;
    if (a > 0 && dk_bit(sc.dk, a - 1) && ix.active[a - 1] >= lo) return w;  // inside a run
    // the run: decode keys from a on, up to the first that leaves (g, s).
    // Its keys hold entries of one (token, kv head) row, so it has at most
    // topk keys (the decode keys of the next sequence follow directly).
    int e = next_non_decode(sc.dk, a, min(n_active, a + P.topk));
    int l = a + 1;
    while (l < e) {
      const int mid = (l + e) >> 1;
      if (ix.active[mid] >= hi) e = mid;
      else l = mid + 1;
    }
    const int len = e - a;
    const int b_last = ix.active[e - 1] - lo;
    const int v_last = si.L - 128 * b_last;
    w.kind = 2;
    w.cnt = len;
    w.n = ceil_div(len, kDecodeBlocks);
    w.adj = (b_last == si.nblk - 1 && v_last < 128) ? (128 - v_last) * P.kvw : 0;
    w.cost = (long long)len * (64 + 128LL * P.kvw) + (long long)w.n * 256 - w.adj;
    return w;
  }
  w.kind = 1;
  w.key = key;
  w.begin = ix.row_ptr[key];
  w.cnt = ix.row_ptr[key + 1] - w.begin;
  w.valid = ix.active_valid[a];
  w.n = ceil_div(w.cnt, P.E);
  const int q = w.cnt / w.n, rem = w.cnt % w.n;
  w.cost = (long long)w.n * (kItemFixed + (long long)w.valid * P.kvw) +
           ((long long)(w.n - rem) * ceil_div(q, P.per_tile) + (long long)rem * ceil_div(q + 1, P.per_tile)) * 256 +
           (long long)w.cnt * P.G * kRowCost;
  return w;
}

__device__ void phase_reduce(const IndexPtrs& ix, const SchedPtrs& sc, const Params& P, unsigned long long* tmp) {
  const int n_active = ix.hdr[kHdrActive], NB = ix.hdr[kHdrNB];
  int lo, hi;
  active_chunk(n_active, &lo, &hi);
  unsigned long long vn = 0, vd = 0;
  for (int a = lo + threadIdx.x; a < hi; a += blockDim.x) {
    const KeyWork w = key_work(ix, sc, P, NB, hi, n_active, a);
    if (w.kind == 1) vn += pack(w.cost, w.n);
    if (w.kind == 2) vd += pack(w.cost, w.n);
  }
  unsigned long long tn, td;
  block_excl_u64(vn, tmp, &tn);
  block_excl_u64(vd, tmp, &td);
  if (threadIdx.x == 0) {
    sc.cta_sums[2 * blockIdx.x] = tn;
    sc.cta_sums[2 * blockIdx.x + 1] = td;
  }
}

__device__ void phase_scan_emit(const IndexPtrs& ix, const SchedPtrs& sc, const Params& P, unsigned long long* tmp) {
  __shared__ KeyWork s_w[kSchTile];
  __shared__ int s_nb[kSchTile], s_db[kSchTile];           // tile-relative item bases
  __shared__ long long s_nc[kSchTile], s_dc[kSchTile];     // global cost bases
  __shared__ int s_tot_n, s_tot_d;
  const int n_active = ix.hdr[kHdrActive], NB = ix.hdr[kHdrNB];
  const unsigned long long kLow = (1ull << kItemBits) - 1;
  // prefix of the chunks before this CTA's, and the totals
  unsigned long long pre_n = 0, pre_d = 0, all_n = 0, all_d = 0;
  for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
    const unsigned long long vn = sc.cta_sums[2 * c], vd = sc.cta_sums[2 * c + 1];
    all_n += vn;
    all_d += vd;
    if (c < (int)blockIdx.x) {
      pre_n += vn;
      pre_d += vd;
    }
  }
  unsigned long long t;
  block_excl_u64(pre_n, tmp, &t); pre_n = t;
  block_excl_u64(pre_d, tmp, &t); pre_d = t;
  block_excl_u64(all_n, tmp, &t); all_n = t;
  block_excl_u64(all_d, tmp, &t); all_d = t;
  const long long Cn = (long long)(all_n >> kItemBits), Cd = (long long)(all_d >> kItemBits);
  const int Nn = (int)(all_n & kLow), Nd = (int)(all_d & kLow);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc.hdr[kSchItems] = Nn;
    sc.hdr[kSchClaim] = 0;
    sc.hdr[kSchExit] = 0;
    sc.hdr[kSchCtas] = P.num_ctas;
    sc.hdr[kSchCostLo] = (int)(Cn & 0xffffffffll);
    sc.hdr[kSchCostHi] = (int)(Cn >> 32);
    sc.hdr[kSchDecItems] = Nd;
    sc.hdr[kSchDecCostLo] = (int)(Cd & 0xffffffffll);
    sc.hdr[kSchDecCostHi] = (int)(Cd >> 32);
    sc.cost_prefix[Nn] = Cn;
    sc.cost_prefix_dec[Nd] = Cd;
    // boundaries whose target is 0 (at least c = 0) start at item 0
    for (int c = 0, e = boundaries_at_or_below(0, Cn, P.num_ctas); c < e; ++c) sc.cta_ptr[c] = 0;
    for (int c = 0, e = boundaries_at_or_below(0, Cd, P.num_ctas); c < e; ++c) sc.cta_ptr_dec[c] = 0;
  }
  int lo, hi;
  active_chunk(n_active, &lo, &hi);
  unsigned long long carry_n = pre_n, carry_d = pre_d;
  for (int t0 = lo; t0 < hi; t0 += kSchTile) {
    unsigned long long vn = 0, vd = 0;
    KeyWork w[kSchPerThread];
#pragma unroll
    for (int j = 0; j < kSchPerThread; ++j) {
      const int a = t0 + threadIdx.x * kSchPerThread + j;
      w[j] = key_work(ix, sc, P, NB, hi, n_active, a);
      if (w[j].kind == 1) vn += pack(w[j].cost, w[j].n);
      if (w[j].kind == 2) vd += pack(w[j].cost, w[j].n);
    }
    unsigned long long tn, td;
    unsigned long long en = block_excl_u64(vn, tmp, &tn);
    unsigned long long ed = block_excl_u64(vd, tmp, &td);
#pragma unroll
    for (int j = 0; j < kSchPerThread; ++j) {
      const int slot = threadIdx.x * kSchPerThread + j;
      s_w[slot] = w[j];
      s_nb[slot] = (int)(en & kLow);
      s_db[slot] = (int)(ed & kLow);
      s_nc[slot] = (long long)((carry_n + en) >> kItemBits);
      s_dc[slot] = (long long)((carry_d + ed) >> kItemBits);
      if (w[j].kind == 1) en += pack(w[j].cost, w[j].n);
      if (w[j].kind == 2) ed += pack(w[j].cost, w[j].n);
    }
    if (threadIdx.x == 0) {
      s_tot_n = (int)(tn & kLow);
      s_tot_d = (int)(td & kLow);
    }
    __syncthreads();
    const int base_n = (int)(carry_n & kLow), base_d = (int)(carry_d & kLow);
    // normal items of the tile
    for (int x = threadIdx.x; x < s_tot_n; x += blockDim.x) {
      int l = 0, h = kSchTile - 1;  // last slot with base <= x holding a normal key
      while (l < h) {
        const int mid = (l + h + 1) >> 1;
        if (s_nb[mid] <= x) l = mid;
        else h = mid - 1;
      }
      while (l > 0 && (s_w[l].kind != 1 || s_nb[l] + s_w[l].n <= x)) --l;
      const KeyWork& k = s_w[l];
      const int i = x - s_nb[l];
      int e0, ne;
      long long pre, cost;
      normal_item(k, P, i, &e0, &ne, &pre, &cost);
      const long long p = s_nc[l] + pre;
      const int item = base_n + x;
      sc.items[item] = make_int4(k.key, k.begin + e0, ne, 0);
      sc.cost_prefix[item] = p;
      for (int c = boundaries_at_or_below(p, Cn, P.num_ctas), e = boundaries_at_or_below(p + cost, Cn, P.num_ctas);
           c < e; ++c)
        sc.cta_ptr[c] = item + 1;
    }
    // decode items of the tile
    for (int x = threadIdx.x; x < s_tot_d; x += blockDim.x) {
      int l = 0, h = kSchTile - 1;
      while (l < h) {
        const int mid = (l + h + 1) >> 1;
        if (s_db[mid] <= x) l = mid;
        else h = mid - 1;
      }
      while (l > 0 && (s_w[l].kind != 2 || s_db[l] + s_w[l].n <= x)) --l;
      const KeyWork& k = s_w[l];
      const int i = x - s_db[l];
      int k0, nk;
      long long pre, cost;
      decode_item(k, P, i, &k0, &nk, &pre, &cost);
      const long long p = s_dc[l] + pre;
      const int item = base_d + x;
      sc.items_dec[item] = make_int4(k.a + k0, ix.row_ptr[ix.active[k.a + k0]], 1, nk);
      sc.cost_prefix_dec[item] = p;
      for (int c = boundaries_at_or_below(p, Cd, P.num_ctas), e = boundaries_at_or_below(p + cost, Cd, P.num_ctas);
           c < e; ++c)
        sc.cta_ptr_dec[c] = item + 1;
    }
    __syncthreads();
    carry_n += tn;
    carry_d += td;
  }
}

struct SchedArgs {
  IndexPtrs ix;
  SchedPtrs sc;
  Params P;
};

__global__ void __launch_bounds__(kSchThreads) k_schedule(SchedArgs a) {
  __shared__ unsigned long long tmp[33];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int* bar = a.sc.hdr + kSchBarCount;
  int epoch = 0;
  int* flags = a.ix.hdr + kHdrFlags;
  phase_flags(a.ix, a.sc, a.P);
  if (!grid_barrier(bar, flags, gridDim.x, epoch)) return;
  phase_reduce(a.ix, a.sc, a.P, tmp);
  if (!grid_barrier(bar, flags, gridDim.x, epoch)) return;
  phase_scan_emit(a.ix, a.sc, a.P, tmp);
}



}  // namespace


static SchedArgs sched_args(const mxsa_problem& p, const IndexPtrs& ix, const SchedPtrs& sc, int num_ctas) {
  const int G = p.num_q_heads / p.num_kv_heads;
  SchedArgs a;
  a.ix = ix;
  a.sc = sc;
  a.P.B = p.num_seqs;
  a.P.Hkv = p.num_kv_heads;
  a.P.G = G;
  a.P.kvw = kv_widened(p) ? 1 : 2;
  a.P.per_tile = std::max(1, MXSA_TILE_ROWS / G);
  a.P.E = MXSA_ITEM_TILES * a.P.per_tile;
  a.P.num_ctas = num_ctas;
  a.P.topk = p.topk;
  return a;
}

cudaError_t launch_schedule(const mxsa_problem& p, const IndexPtrs& ix, const SchedPtrs& sc,
                            const mxsa_sched_layout& lay, int num_ctas, cudaStream_t st) {
  (void)lay;
  SchedArgs a = sched_args(p, ix, sc, num_ctas);
  const int grid = coop_grid(reinterpret_cast<const void*>(k_schedule), kSchThreads);
  if (grid <= 0) return cudaErrorNotSupported;
  cudaError_t e = cudaMemsetAsync(sc.hdr, 0, kSchInts * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_schedule), dim3(grid), dim3(kSchThreads), args,
                                     0, st);
}

}  // namespace mxsa
