// Index build and schedule fused into one cooperative launch (mxsa_plan).
// The result is the same index as mxsa_build_index and the same two work
// lists as mxsa_schedule; the schedule is folded into the index's own scan:
//
//   seq + zero   every CTA recomputes the per-sequence scan (B <= 1024; one
//                CTA and a barrier otherwise), CTA 0 stores it; every CTA
//                fills its share of the token map and clears counters and
//                bitmap rows                                   -> barrier
//   mark         one warp per (token, kv head) row, as in the index build;
//                it also records the row's entry count and its smallest and
//                largest selected block                        -> barrier
//   reduce       one contiguous chunk of keys per CTA; each key adds to
//                three sums: (entries, key active), (normal items, cost),
//                (decode items, cost).  A decode key (single-token sequence)
//                contributes its whole run when its block is the row's
//                smallest; the run length is the row's entry count and the
//                partial-last-block adjustment applies when the row's
//                largest block is the sequence's last      -> barrier
//   scan + emit  each CTA adds the sums of the chunks before it; per tile of
//                256 keys: row_ptr, the active-key list, the entries (bitmap
//                walk), and the items of both lists with their cost prefixes
//                and CTA boundaries.  A decode run's keys each hold one
//                entry, so the entry of its k-th key is the first key's + k.
#include <algorithm>

#include "index_phases.cuh"
#include "sched_common.cuh"

namespace mxsa {

namespace {

using namespace sch;

constexpr int kPlanThreads = 256;
constexpr int kPlanTile = 256;  // keys per scan tile: one per thread
constexpr int kRedundantSeqMax = 1024;
static_assert(kPlanThreads == ixp::kIndexThreads, "index phases run with the same block size");

struct PlanArgs {
  ixp::IndexArgs ia;
  SchedPtrs sc;
  Params P;
};

// schedule contribution of key `key` (kv head g, block b of the sequence
// si) with `c` entries (kind 0: none)
__device__ __forceinline__ KeyWork plan_key_work(const IndexPtrs& ix, const Params& P, int key, int g,
                                                 const SeqInfo& si, int b, int c) {
  KeyWork w{};
  if (c == 0) return w;
  if (P.G <= kDecodeMaxG && si.tq == 1) {
    const int row = si.q_begin * P.Hkv + g;
    if (b != ix.row_minb[row]) return w;  // not the first key of its run
    const int len = ix.row_nnz[row];
    const int bmax = ix.row_maxb[row];
    const int v_last = si.L - 128 * bmax;
    w.kind = 2;
    w.cnt = len;
    w.n = ceil_div(len, kDecodeBlocks);
    w.adj = (bmax == si.nblk - 1 && v_last < 128) ? (128 - v_last) * P.kvw : 0;
    w.cost = (long long)len * (64 + 128LL * P.kvw) + (long long)w.n * 256 - w.adj;
    return w;
  }
  w.kind = 1;
  w.key = key;
  w.cnt = c;
  const int valid = si.L - 128 * b;
  w.valid = valid < 128 ? valid : 128;
  w.n = ceil_div(c, P.E);
  const int q = c / w.n, rem = c % w.n;
  w.cost = (long long)w.n * (kItemFixed + (long long)w.valid * P.kvw) +
           ((long long)(w.n - rem) * ceil_div(q, P.per_tile) + (long long)rem * ceil_div(q + 1, P.per_tile)) * 256 +
           (long long)c * P.G * kRowCost;
  return w;
}

// reduce: each key's entry count is the population of its bitmap row (the
// mark phase does not count), stored for the scan; then the three sums
__device__ __forceinline__ void plan_reduce(const IndexPtrs& ix, const Params& P, const ixp::SeqTab& tab,
                                            unsigned long long* tmp) {
  const int n_keys = ix.hdr[kHdrKeys], NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW];
  int lo, hi;
  ixp::key_chunk(n_keys, &lo, &hi);
  unsigned long long vi = 0, vn = 0, vd = 0;
  for (int k = lo + threadIdx.x; k < hi; k += blockDim.x) {
    const int g = k / NB, r = k - g * NB;
    const SeqInfo si = tab.get(tab.find(r));
    const int b = r - si.blk_off;
    const uint32_t* row = ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words;
    int c = 0;
    for (int w = 0; w < si.words; ++w) c += __popc(row[w]);
    ix.counts[k] = c;
    vi += ixp::key_payload(c);
    const KeyWork w = plan_key_work(ix, P, k, g, si, b, c);
    if (w.kind == 1) vn += pack(w.cost, w.n);
    if (w.kind == 2) vd += pack(w.cost, w.n);
  }
  U3 tot;
  block_excl_u64x3(U3{vi, vn, vd}, tmp, &tot);
  if (threadIdx.x == 0) {
    ix.cta_sums[3 * blockIdx.x] = tot.x;
    ix.cta_sums[3 * blockIdx.x + 1] = tot.y;
    ix.cta_sums[3 * blockIdx.x + 2] = tot.z;
  }
}

__device__ __forceinline__ void plan_scan_emit(const IndexPtrs& ix, const SchedPtrs& sc, const Params& P, int Hkv,
                                               int topk, const ixp::SeqTab& tab, unsigned long long* tmp) {
  __shared__ KeyWork s_w[kPlanTile];
  __shared__ int s_nb[kPlanTile], s_db[kPlanTile];
  __shared__ long long s_nc[kPlanTile], s_dc[kPlanTile];
  __shared__ int s_long_key[kPlanTile], s_long_base[kPlanTile];
  __shared__ int s_n_long, s_tot_n, s_tot_d;
  const int n_keys = ix.hdr[kHdrKeys], NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const int warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  const unsigned long long kLow31 = (1ull << 31) - 1, kLow = (1ull << kItemBits) - 1;
  // prefixes of the chunks before this CTA and the totals, all three sums
  unsigned long long pi = 0, pn = 0, pd = 0, ai = 0, an = 0, ad = 0;
  for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
    const unsigned long long vi = ix.cta_sums[3 * c], vn = ix.cta_sums[3 * c + 1], vd = ix.cta_sums[3 * c + 2];
    ai += vi;
    an += vn;
    ad += vd;
    if (c < (int)blockIdx.x) {
      pi += vi;
      pn += vn;
      pd += vd;
    }
  }
  U3 t3;
  block_excl_u64x3(U3{pi, pn, pd}, tmp, &t3);
  pi = t3.x;
  pn = t3.y;
  pd = t3.z;
  block_excl_u64x3(U3{ai, an, ad}, tmp, &t3);
  ai = t3.x;
  an = t3.y;
  ad = t3.z;
  const long long Cn = (long long)(an >> kItemBits), Cd = (long long)(ad >> kItemBits);
  const int Nn = (int)(an & kLow), Nd = (int)(ad & kLow);
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    ix.row_ptr[n_keys] = (int)(ai >> 31);
    ix.hdr[kHdrNnz] = (int)(ai >> 31);
    ix.hdr[kHdrActive] = (int)(ai & kLow31);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc.hdr[kSchItems] = Nn;
    sc.hdr[kSchCtas] = P.num_ctas;
    sc.hdr[kSchClaim] = 0;
    sc.hdr[kSchExit] = 0;
    sc.hdr[kSchCostLo] = (int)(Cn & 0xffffffffll);
    sc.hdr[kSchCostHi] = (int)(Cn >> 32);
    sc.hdr[kSchDecItems] = Nd;
    sc.hdr[kSchDecCostLo] = (int)(Cd & 0xffffffffll);
    sc.hdr[kSchDecCostHi] = (int)(Cd >> 32);
    sc.cost_prefix[Nn] = Cn;
    sc.cost_prefix_dec[Nd] = Cd;
    for (int c = 0, e = boundaries_at_or_below(0, Cn, P.num_ctas); c < e; ++c) sc.cta_ptr[c] = 0;
    for (int c = 0, e = boundaries_at_or_below(0, Cd, P.num_ctas); c < e; ++c) sc.cta_ptr_dec[c] = 0;
  }
  int lo, hi;
  ixp::key_chunk(n_keys, &lo, &hi);
  unsigned long long ci = pi, cn = pn, cd = pd;
  for (int t0 = lo; t0 < hi; t0 += kPlanTile) {
    const int key = t0 + threadIdx.x;
    const int c = key < hi ? ix.counts[key] : 0;
    const int g = key / NB, r = key - g * NB;
    SeqInfo si{};
    if (c > 0) si = tab.get(tab.find(r));
    const int b = r - si.blk_off;
    KeyWork w = plan_key_work(ix, P, key, g, si, b, c);
    if (threadIdx.x == 0) s_n_long = 0;
    U3 tt;
    const U3 ex = block_excl_u64x3(U3{ixp::key_payload(c), w.kind == 1 ? pack(w.cost, w.n) : 0ull,
                                      w.kind == 2 ? pack(w.cost, w.n) : 0ull},
                                   tmp, &tt);
    const unsigned long long ei = ex.x, en = ex.y, ed = ex.z;
    const unsigned long long ti = tt.x, tn = tt.y, td = tt.z;
    const unsigned long long run = ci + ei;
    if (key < hi) {
      const int base = (int)(run >> 31);
      ix.row_ptr[key] = base;
      w.begin = base;
      if (c > 0) {
        const int pos = (int)(run & kLow31);
        w.a = pos;
        ix.active[pos] = key;
        const int valid = si.L - 128 * b;
        ix.active_valid[pos] = valid < 128 ? valid : 128;
        if (si.words <= 2) {
          ixp::emit_row_serial(ix, ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words, si.words,
                               ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq, si.q_begin, g,
                               Hkv, topk, base);
        } else {
          const int at = atomicAdd(&s_n_long, 1);
          s_long_key[at] = key;
          s_long_base[at] = base;
        }
      }
    }
    s_w[threadIdx.x] = w;
    s_nb[threadIdx.x] = (int)(en & kLow);
    s_db[threadIdx.x] = (int)(ed & kLow);
    s_nc[threadIdx.x] = (long long)((cn + en) >> kItemBits);
    s_dc[threadIdx.x] = (long long)((cd + ed) >> kItemBits);
    if (threadIdx.x == 0) {
      s_tot_n = (int)(tn & kLow);
      s_tot_d = (int)(td & kLow);
    }
    __syncthreads();
    // long bitmap rows: one warp per key, or, when the tile has at most half
    // as many long rows as warps (a few popular keys), several warps per key
    const int wpr = s_n_long > 0 && 2 * s_n_long <= n_warps ? n_warps / s_n_long : 1;
    for (int i = warp / wpr; i < s_n_long; i += n_warps / wpr) {
      const int k2 = s_long_key[i];
      const int g = k2 / NB, r = k2 - g * NB;
      const SeqInfo si = tab.get(tab.find(r));
      const int b = r - si.blk_off;
      const uint32_t* bm = ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words;
      const uint8_t* km = ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq;
      if (wpr == 1)
        ixp::emit_row_warp(ix, bm, si.words, km, si.q_begin, g, Hkv, topk, s_long_base[i]);
      else
        ixp::emit_row_shared(ix, bm, si.words, km, si.q_begin, g, Hkv, topk, s_long_base[i], warp % wpr, wpr);
    }
    const int base_n = (int)(cn & kLow), base_d = (int)(cd & kLow);
    for (int x = threadIdx.x; x < s_tot_n; x += blockDim.x) {
      int l = 0, h = kPlanTile - 1;  // last slot whose item base is <= x
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
      for (int c2 = boundaries_at_or_below(p, Cn, P.num_ctas), e = boundaries_at_or_below(p + cost, Cn, P.num_ctas);
           c2 < e; ++c2)
        sc.cta_ptr[c2] = item + 1;
    }
    for (int x = threadIdx.x; x < s_tot_d; x += blockDim.x) {
      int l = 0, h = kPlanTile - 1;
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
      sc.items_dec[item] = make_int4(k.a + k0, k.begin + k0, 1, nk);
      sc.cost_prefix_dec[item] = p;
      for (int c2 = boundaries_at_or_below(p, Cd, P.num_ctas), e = boundaries_at_or_below(p + cost, Cd, P.num_ctas);
           c2 < e; ++c2)
        sc.cta_ptr_dec[c2] = item + 1;
    }
    __syncthreads();
    ci += ti;
    cn += tn;
    cd += td;
  }
}

// ------------------------------------------------------------------------
// All-decode batches (every sequence has at most one new token, G <= 16):
// every selected key then holds exactly one entry, so entries, active keys
// and decode runs all follow the (kv head, sequence) rows in key order and
// the whole plan needs one grid barrier.  The result is the same index and
// schedule as the general phases.
//
//   A  one warp per row (g, s) of the CTA's share: validate the row's
//      selections (range, duplicates), rank the distinct blocks, park the
//      ranked (block, slot) list in the row's own slot_entry range, and sum
//      entries, decode items and cost per CTA               -> barrier
//   B  CTA prefixes; per row: slot_entry, entries, active keys, row_ptr of
//      every key of the row, and the row's decode items with their cost
//      prefixes and CTA boundaries.
constexpr int kFastRowsChunk = kPlanThreads;

__device__ __forceinline__ void fast_rows(int n_rows, int* r0, int* r1) {
  *r0 = (int)((long long)blockIdx.x * n_rows / gridDim.x);
  *r1 = (int)((long long)(blockIdx.x + 1) * n_rows / gridDim.x);
}

// adj of a decode run: cost removed for the unread tail of a partial last block
__device__ __forceinline__ int fast_adj(const SeqInfo& si, int bmax, int kvw) {
  if (bmax < 0 || bmax != si.nblk - 1) return 0;
  const int v_last = si.L - 128 * bmax;
  return v_last < 128 ? (128 - v_last) * kvw : 0;
}

__device__ __forceinline__ void fast_phase_a(const IndexPtrs& ix, const int32_t* sel, const Params& P,
                                             const ixp::SeqTab& tab, int topk, int32_t (*rowbuf)[256],
                                             unsigned long long* tmp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int n_rows = P.Hkv * P.B;
  int r0, r1;
  fast_rows(n_rows, &r0, &r1);
  const long long per_key = 64 + 128LL * P.kvw;
  unsigned long long se = 0, sit = 0, scost = 0;
  int flags = 0;
  for (int R = r0 + w; R < r1; R += nw) {
    const int g = R / P.B, s = R - g * P.B;
    const SeqInfo si = tab.get(s);
    if (si.tq != 1) continue;  // uniform per warp
    const int row = si.q_begin * P.Hkv + g;
    const long long base_slot = (long long)row * topk;
    for (int k = lane; k < topk; k += 32) rowbuf[w][k] = sel[base_slot + k];
    __syncwarp();
    // validity of each slot: a block of the sequence, not repeated earlier
    // in the row (the first occurrence is kept)
    bool ok[8];
    int nv = 0, bmax = -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = lane + 32 * u;
      ok[u] = false;
      if (k >= topk) continue;
      const int b = rowbuf[w][k];
      if (b == -1) continue;
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
      ok[u] = true;
      ++nv;
      bmax = max(bmax, b);
    }
    __syncwarp();
    // invalid slots out of the ranking
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = lane + 32 * u;
      if (k < topk && !ok[u]) rowbuf[w][k] = 0x7fffffff;
    }
    __syncwarp();
    // rank = distinct valid blocks below: the row's blocks in ascending order
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = lane + 32 * u;
      if (k >= topk || !ok[u]) continue;
      const int b = rowbuf[w][k];
      int rank = 0;
      for (int k2 = 0; k2 < topk; ++k2) rank += rowbuf[w][k2] < b;
      ix.slot_entry[base_slot + rank] = (b << 8) | k;
    }
    const int nnz = __reduce_add_sync(0xffffffffu, nv);
    bmax = __reduce_max_sync(0xffffffffu, bmax);
    if (lane == 0) {
      ix.row_nnz[row] = nnz;
      ix.row_maxb[row] = bmax;
      const int items = ceil_div(nnz, kDecodeBlocks);
      se += nnz;
      sit += items;
      scost += nnz ? (unsigned long long)(nnz * per_key + (long long)items * 256 - fast_adj(si, bmax, P.kvw)) : 0ull;
    }
    __syncwarp();
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(&ix.hdr[kHdrFlags], flags);
  U3 tot;
  block_excl_u64x3(U3{se, sit, scost}, tmp, &tot);
  if (threadIdx.x == 0) {
    ix.cta_sums[3 * blockIdx.x] = tot.x;
    ix.cta_sums[3 * blockIdx.x + 1] = tot.y;
    ix.cta_sums[3 * blockIdx.x + 2] = tot.z;
  }
}

__device__ __forceinline__ void fast_phase_b(const IndexPtrs& ix, const SchedPtrs& sc, const Params& P,
                                             const ixp::SeqTab& tab, int total_q, int topk, int32_t (*rowbuf)[256],
                                             unsigned long long* tmp) {
  __shared__ unsigned long long s_base[3][kFastRowsChunk];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int NB = ix.hdr[kHdrNB], n_keys = ix.hdr[kHdrKeys];
  const int n_rows = P.Hkv * P.B;
  // this CTA's prefixes and the totals
  unsigned long long pe = 0, pit = 0, pc = 0, ae = 0, ait = 0, ac = 0;
  for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
    const unsigned long long e = ix.cta_sums[3 * c], it = ix.cta_sums[3 * c + 1], co = ix.cta_sums[3 * c + 2];
    ae += e;
    ait += it;
    ac += co;
    if (c < (int)blockIdx.x) {
      pe += e;
      pit += it;
      pc += co;
    }
  }
  U3 t3;
  block_excl_u64x3(U3{pe, pit, pc}, tmp, &t3);
  pe = t3.x;
  pit = t3.y;
  pc = t3.z;
  block_excl_u64x3(U3{ae, ait, ac}, tmp, &t3);
  const int E = (int)t3.x, Nd = (int)t3.y;
  const long long Cd = (long long)t3.z;
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    ix.row_ptr[n_keys] = E;
    ix.hdr[kHdrNnz] = E;
    ix.hdr[kHdrActive] = E;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc.hdr[kSchItems] = 0;
    sc.hdr[kSchCtas] = P.num_ctas;
    sc.hdr[kSchClaim] = 0;
    sc.hdr[kSchExit] = 0;
    sc.hdr[kSchCostLo] = 0;
    sc.hdr[kSchCostHi] = 0;
    sc.hdr[kSchDecItems] = Nd;
    sc.hdr[kSchDecCostLo] = (int)(Cd & 0xffffffffll);
    sc.hdr[kSchDecCostHi] = (int)(Cd >> 32);
    sc.cost_prefix[0] = 0;
    sc.cost_prefix_dec[Nd] = Cd;
    for (int c = 0; c <= P.num_ctas; ++c) sc.cta_ptr[c] = 0;
    for (int c = 0, e = boundaries_at_or_below(0, Cd, P.num_ctas); c < e; ++c) sc.cta_ptr_dec[c] = 0;
  }
  // tokens outside every decode row (only when cu_seqlens_q was invalid):
  // their slots index nothing
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total_q;
       t += (long long)gridDim.x * blockDim.x) {
    if (tab.get(ix.token_seq[t]).tq == 1) continue;
    for (long long x = t * P.Hkv * topk; x < (t + 1) * P.Hkv * topk; ++x) ix.slot_entry[x] = -1;
  }
  int r0, r1;
  fast_rows(n_rows, &r0, &r1);
  unsigned long long ce = pe, cit = pit, cc = pc;
  for (int c0 = r0; c0 < r1; c0 += kFastRowsChunk) {
    // per-row bases of this chunk (rows in key order)
    const int R = c0 + threadIdx.x;
    unsigned long long ve = 0, vit = 0, vc = 0;
    if (R < r1) {
      const int g = R / P.B, s = R - g * P.B;
      const SeqInfo si = tab.get(s);
      if (si.tq == 1) {
        const int row = si.q_begin * P.Hkv + g;
        const int nnz = ix.row_nnz[row];
        const int items = ceil_div(nnz, kDecodeBlocks);
        ve = nnz;
        vit = items;
        vc = nnz ? (unsigned long long)(nnz * (64 + 128LL * P.kvw) + (long long)items * 256 -
                                        fast_adj(si, ix.row_maxb[row], P.kvw))
                 : 0ull;
      }
    }
    U3 tt;
    const U3 ex = block_excl_u64x3(U3{ve, vit, vc}, tmp, &tt);
    s_base[0][threadIdx.x] = ce + ex.x;
    s_base[1][threadIdx.x] = cit + ex.y;
    s_base[2][threadIdx.x] = cc + ex.z;
    __syncthreads();
    const int nr = min(kFastRowsChunk, r1 - c0);
    for (int rr = w; rr < nr; rr += nw) {
      const int Rw = c0 + rr;
      const int g = Rw / P.B, s = Rw - g * P.B;
      const SeqInfo si = tab.get(s);
      const int base_e = (int)s_base[0][rr];
      const int base_it = (int)s_base[1][rr];
      const long long base_c = (long long)s_base[2][rr];
      const long long key0 = (long long)g * NB + si.blk_off;
      int nnz = 0, bmax = -1;
      if (si.tq == 1) {
        const int row = si.q_begin * P.Hkv + g;
        const long long base_slot = (long long)row * topk;
        nnz = ix.row_nnz[row];
        bmax = ix.row_maxb[row];
        for (int j = lane; j < nnz; j += 32) rowbuf[w][j] = ix.slot_entry[base_slot + j];
        __syncwarp();
        for (int k = lane; k < topk; k += 32) ix.slot_entry[base_slot + k] = -1;
        __syncwarp();
        for (int j = lane; j < nnz; j += 32) {
          const int v = rowbuf[w][j], b = v >> 8, k = v & 255;
          const int pos = base_e + j;
          ix.active[pos] = (int)(key0 + b);
          ix.active_valid[pos] = min(128, si.L - 128 * b);
          ix.entries[pos] = (int)(base_slot + k);
          ix.slot_entry[base_slot + k] = pos;
        }
      }
      __syncwarp();
      // row_ptr of every key of the row: entries before it.  Windows of 32
      // blocks: `cur` ranked blocks lie below the window, and those inside
      // it (at most 32) are the ranks that follow, so one look at ranks
      // cur .. cur + 31 gives the window's bit mask.
      for (int b0 = 0, cur = 0; b0 < si.nblk; b0 += 32) {
        const int jr = cur + lane;
        const int bj = jr < nnz ? (rowbuf[w][jr] >> 8) : 0x7fffffff;
        const bool in = bj < b0 + 32;
        const unsigned mask = __reduce_or_sync(0xffffffffu, in ? 1u << (bj - b0) : 0u);
        if (b0 + lane < si.nblk) ix.row_ptr[key0 + b0 + lane] = base_e + cur + __popc(mask & ((1u << lane) - 1));
        cur += __popc(__ballot_sync(0xffffffffu, in));
      }
      // the row's decode items
      if (nnz > 0) {
        KeyWork kw{};
        kw.kind = 2;
        kw.a = base_e;
        kw.begin = base_e;
        kw.cnt = nnz;
        kw.n = ceil_div(nnz, kDecodeBlocks);
        kw.adj = fast_adj(si, bmax, P.kvw);
        for (int i = lane; i < kw.n; i += 32) {
          int k0, nk;
          long long pre, cost;
          decode_item(kw, P, i, &k0, &nk, &pre, &cost);
          const long long pfx = base_c + pre;
          const int item = base_it + i;
          sc.items_dec[item] = make_int4(kw.a + k0, kw.begin + k0, 1, nk);
          sc.cost_prefix_dec[item] = pfx;
          for (int c2 = boundaries_at_or_below(pfx, Cd, P.num_ctas),
                   e = boundaries_at_or_below(pfx + cost, Cd, P.num_ctas);
               c2 < e; ++c2)
            sc.cta_ptr_dec[c2] = item + 1;
        }
      }
      __syncwarp();
    }
    ce += tt.x;
    cit += tt.y;
    cc += tt.z;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kPlanThreads, 2) k_plan(PlanArgs a) {
  __shared__ unsigned long long tmp[3 * 33];
  __shared__ int32_t rowbuf[ixp::kMarkWarps][256];
  __shared__ int s_tab[6][ixp::kSeqTab];
  pdl_launch_dependents();
  const ixp::IndexArgs& ia = a.ia;
  int* bar = ia.ix.hdr + kHdrBarCount;
  int epoch = 0;
  int* flags = ia.ix.hdr + kHdrFlags;
  const unsigned nb = gridDim.x;
  ixp::SeqTotals tot;
  if (ia.B <= kRedundantSeqMax) {
    tot = ixp::phase_seq(ia.ix, ia.cu, ia.lens, ia.B, ia.total_q, ia.Hkv, ia.cap_len, ia.causal,
                         reinterpret_cast<long long*>(tmp), blockIdx.x == 0, s_tab);
  } else {
    if (blockIdx.x == 0)
      ixp::phase_seq(ia.ix, ia.cu, ia.lens, ia.B, ia.total_q, ia.Hkv, ia.cap_len, ia.causal,
                     reinterpret_cast<long long*>(tmp));
    if (!grid_barrier(bar, flags, nb, epoch)) return;
    tot = ixp::SeqTotals{ia.ix.hdr[kHdrNB], ia.ix.hdr[kHdrBMW], ia.ix.hdr[kHdrKMW]};
  }
  ixp::phase_token_seq(ia.ix, ia.cu, ia.B, ia.total_q, ia.B <= ixp::kSeqTab ? s_tab[3] : nullptr);
  // (block << 8 | slot) of the ranked rows must fit an int: blocks < 2^23
  if (ia.B <= ixp::kSeqTab && a.P.G <= kDecodeMaxG && ia.cap_len < (1 << 30)) {
    // all-decode batch (every sequence at most one new token): one barrier
    bool all_decode = true;
    for (int s = threadIdx.x; s < ia.B; s += blockDim.x) all_decode &= s_tab[5][s] <= 1;
    if (__syncthreads_and(all_decode)) {
      const ixp::SeqTab tab{ia.ix.seq, s_tab, ia.B};
      fast_phase_a(ia.ix, ia.sel, a.P, tab, ia.topk, rowbuf, tmp);
      if (!grid_barrier(bar, flags, nb, epoch)) return;
      fast_phase_b(ia.ix, a.sc, a.P, tab, ia.total_q, ia.topk, rowbuf, tmp);
      return;
    }
  }
  ixp::phase_zero(ia.ix, ia.Hkv, tot, false);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  ixp::phase_mark(ia.ix, ia.sel, ia.total_q, ia.Hkv, ia.topk, ia.causal, rowbuf, false);
  const ixp::SeqTab tab{ia.ix.seq, ia.B <= ixp::kSeqTab ? s_tab : nullptr, ia.B};
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  plan_reduce(ia.ix, a.P, tab, tmp);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  plan_scan_emit(ia.ix, a.sc, a.P, ia.Hkv, ia.topk, tab, tmp);
}

}  // namespace


cudaError_t launch_plan(const mxsa_problem& p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                        const IndexPtrs& ix, const SchedPtrs& sc, int num_ctas, cudaStream_t st) {
  PlanArgs a;
  a.ia = ixp::IndexArgs{ix, sel, cu, lens, p.num_seqs, p.total_q, p.num_kv_heads, p.topk,
                        p.max_pages_per_seq * p.page_size, p.causal};
  a.sc = sc;
  const int G = p.num_q_heads / p.num_kv_heads;
  a.P.B = p.num_seqs;
  a.P.Hkv = p.num_kv_heads;
  a.P.G = G;
  a.P.kvw = kv_widened(p) ? 1 : 2;
  a.P.per_tile = std::max(1, MXSA_TILE_ROWS / G);
  a.P.E = MXSA_ITEM_TILES * a.P.per_tile;
  a.P.num_ctas = num_ctas;
  a.P.topk = p.topk;
  const int grid = coop_grid(reinterpret_cast<const void*>(k_plan), kPlanThreads);
  if (grid <= 0) return cudaErrorNotSupported;
  cudaError_t e = cudaMemsetAsync(ix.hdr, 0, kHdrInts * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_plan), dim3(grid), dim3(kPlanThreads), args, 0,
                                     st);
}

}  // namespace mxsa

#ifdef MXSA_TEST_HOOKS
// Test builds only: makes CTA `cta` of the next plan launches skip its
// arrival at grid barrier number `barrier` (1 = the first); cta = -1 turns
// the switch off.  Synchronous.
extern "C" mxsa_status mxsa_test_skip_barrier_arrival(int32_t cta, int32_t barrier) {
  if (cudaMemcpyToSymbol(mxsa::g_skip_cta, &cta, sizeof(cta)) != cudaSuccess) return MXSA_ERR_CUDA;
  if (cudaMemcpyToSymbol(mxsa::g_skip_barrier, &barrier, sizeof(barrier)) != cudaSuccess) return MXSA_ERR_CUDA;
  return MXSA_OK;
}
#endif
