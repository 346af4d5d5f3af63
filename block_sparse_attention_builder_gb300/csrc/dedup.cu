// Index builder with cross-sequence block dedup (mxsa_build_index_dedup).
// The README of fw-ai/minimax-kernels (intro) makes the KV block the unit
// that is loaded once for every query that selected it; sequences that share
// a cached prefix point their block tables at the same physical pages, so
// such a block is keyed by its pages here, and its rows of every sequence
// meet in one key:
//
//   a block (s, b) is shareable when it is full (128 b + 128 <= L_s) and its
//   pages lie in [0, num_pages); owner(s, b) = the smallest sequence whose
//   block b is shareable with the same pages (a block that is not shareable
//   owns itself); the rows of (s, b) join key g * NB + blk_off[owner] + b.
//
// Within a key the entries stay in slot order.  Slots grow with the token
// and a sequence's tokens precede the next sequence's, so a key's entries
// are its member blocks' own rows (bitmap walks, as in the plain build)
// taken in sequence order.
//
// One cooperative launch, seven phases separated by bounded grid barriers:
//   seq     CTA 0: per-sequence scan; every CTA: token -> sequence map and
//           the page array set to "none"
//   zero    counters and bitmaps cleared; every shareable block offers its
//           packed (b, s) to its first page's slot with a 64-bit atomicMin
//   mark    the plain build's mark phase (bitmap rows per (g, s, b)); every
//           block finds its owner: the page slot's (b, s) when it has the
//           same b and pages (then it is the smallest such sequence), else a
//           search over the smaller sequences (pages reused at another
//           logical block, or 64-token page pairs that share only one page);
//           each owner block counts its members
//   fold    per block, each head's row population is kept as its own count
//           and added to its owner's key; owner blocks with other members
//           are listed and given room for their member list
//   reduce  per-CTA sums of the key counts (the plain build's phase); one
//           warp per listed owner block walks the sequences from the owner
//           up (32 lanes x 4 at a time) and writes its members in order
//   scan    row_ptr, active keys and the entries of keys that are their
//           block's only member (as in the plain build); keys of listed
//           owner blocks are queued with their first entry
//   group   one warp per queued key writes its entries: its members' own
//           bitmap rows in member order
// The last two phases spread the shared blocks' work over the whole grid:
// their keys lie in a few sequences' key ranges, which the scan's chunks
// would otherwise leave to a few CTAs.
#include "index_phases.cuh"

namespace mxsa {

namespace {

using ixp::kIndexThreads;

struct DedupArgs {
  ixp::IndexArgs ia;
  DedupPtrs d;
  const int32_t* bt;
  int max_pages, num_pages, ps;
};

// Pages of block b of sequence s (metadata si) when the block is shareable:
// full, and every page inside [0, num_pages).  A full block lies inside the
// block-table row, since L_s <= max_pages * page_size.
__device__ __forceinline__ bool shareable(const DedupArgs& a, const SeqInfo& si, int s, int b, int* p0, int* p1) {
  if (128LL * b + 128 > si.L) return false;
  const int32_t* row = a.bt + (size_t)s * a.max_pages;
  if (a.ps == 128) {
    *p0 = row[b];
    *p1 = -1;
    return *p0 >= 0 && *p0 < a.num_pages;
  }
  *p0 = row[2 * b];
  *p1 = row[2 * b + 1];
  return *p0 >= 0 && *p0 < a.num_pages && *p1 >= 0 && *p1 < a.num_pages;
}

__device__ __forceinline__ unsigned long long pack_bs(int b, int s) {
  return ((unsigned long long)(unsigned)b << 32) | (unsigned)s;
}

__device__ __forceinline__ long long grid_tid() { return (long long)blockIdx.x * blockDim.x + threadIdx.x; }
__device__ __forceinline__ long long grid_threads() { return (long long)gridDim.x * blockDim.x; }

__device__ void phase_offer(const DedupArgs& a) {
  const IndexPtrs& ix = a.ia.ix;
  const int NB = ix.hdr[kHdrNB];
  for (long long r = grid_tid(); r < NB; r += grid_threads()) {
    a.d.gsize[r] = 0;
    const int s = ixp::seq_of_block(ix.seq, a.ia.B, (int)r);
    const SeqInfo si = ix.seq[s];
    const int b = (int)r - si.blk_off;
    int p0, p1;
    if (shareable(a, si, s, b, &p0, &p1)) atomicMin(&a.d.page_min[p0], pack_bs(b, s));
  }
}

__device__ void phase_owner(const DedupArgs& a) {
  const IndexPtrs& ix = a.ia.ix;
  const int NB = ix.hdr[kHdrNB];
  for (long long r = grid_tid(); r < NB; r += grid_threads()) {
    const int s = ixp::seq_of_block(ix.seq, a.ia.B, (int)r);
    const SeqInfo si = ix.seq[s];
    const int b = (int)r - si.blk_off;
    int o = s, p0, p1;
    if (shareable(a, si, s, b, &p0, &p1)) {
      const unsigned long long c = a.d.page_min[p0];
      const int cb = (int)(c >> 32), cs = (int)(c & 0xffffffffull);
      if (cb == b && (a.ps == 128 || a.bt[(size_t)cs * a.max_pages + 2 * b + 1] == p1)) {
        o = cs;
      } else {
        for (int s2 = 0; s2 < s; ++s2) {
          int q0, q1;
          if (shareable(a, ix.seq[s2], s2, b, &q0, &q1) && q0 == p0 && q1 == p1) {
            o = s2;
            break;
          }
        }
      }
    }
    a.d.owner[r] = o;
    atomicAdd(&a.d.gsize[ix.seq[o].blk_off + b], 1);
  }
}

constexpr int kFoldHeads = 8;
__device__ void phase_fold(const DedupArgs& a) {
  const IndexPtrs& ix = a.ia.ix;
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW];
  for (long long r = grid_tid(); r < NB; r += grid_threads()) {
    const int s = ixp::seq_of_block(ix.seq, a.ia.B, (int)r);
    const SeqInfo si = ix.seq[s];
    const int b = (int)r - si.blk_off;
    const int orow = ix.seq[a.d.owner[r]].blk_off + b;
    // the heads' rows kFoldHeads at a time: their bitmap reads are issued
    // together, then the counts are stored
    for (int g0 = 0; g0 < a.ia.Hkv; g0 += kFoldHeads) {
      int c[kFoldHeads];
#pragma unroll
      for (int u = 0; u < kFoldHeads; ++u) {
        const int g = g0 + u;
        c[u] = 0;
        if (g < a.ia.Hkv) {
          const uint32_t* row = ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words;
          if (si.words == 1) c[u] = __popc(row[0]);
          else
            for (int w = 0; w < si.words; ++w) c[u] += __popc(row[w]);
        }
      }
#pragma unroll
      for (int u = 0; u < kFoldHeads; ++u) {
        const int g = g0 + u;
        if (g < a.ia.Hkv) {
          a.d.own_count[(long long)g * NB + r] = c[u];
          if (c[u] > 0) atomicAdd(&ix.counts[(long long)g * NB + orow], c[u]);
        }
      }
    }
    const int m = a.d.gsize[r];
    if (m > 1) {
      a.d.glist[atomicAdd(&ix.hdr[kHdrGroups], 1)] = (int)r;
      a.d.mbeg[r] = atomicAdd(&ix.hdr[kHdrMembers], m);
    }
  }
}

// One warp writes the member sequences of owner block R (sequence o, block
// b) in increasing order: the sequences s >= o with owner(s, b) == o.
constexpr int kWalkUnroll = 4;
__device__ void walk_members(const DedupArgs& a, int R) {
  const IndexPtrs& ix = a.ia.ix;
  const int lane = threadIdx.x & 31;
  const int o = ixp::seq_of_block(ix.seq, a.ia.B, R);
  const int b = R - ix.seq[o].blk_off;
  const int m = a.d.gsize[R];
  int32_t* out = a.d.mlist + a.d.mbeg[R];
  int found = 0;
  for (int s0 = o; s0 < a.ia.B && found < m; s0 += 32 * kWalkUnroll) {
    bool mem[kWalkUnroll];
#pragma unroll
    for (int u = 0; u < kWalkUnroll; ++u) {
      const int s = s0 + 32 * u + lane;
      mem[u] = false;
      if (s < a.ia.B) {
        const int nblk = ix.seq[s].nblk, boff = ix.seq[s].blk_off;
        mem[u] = b < nblk && a.d.owner[boff + b] == o;
      }
    }
#pragma unroll
    for (int u = 0; u < kWalkUnroll; ++u) {
      const unsigned bal = __ballot_sync(0xffffffffu, mem[u]);
      if (mem[u]) out[found + __popc(bal & ((1u << lane) - 1u))] = s0 + 32 * u + lane;
      found += __popc(bal);
    }
  }
}

// One warp writes the entries of key (g, owner block R) from `base`: the
// members' own bitmap rows in member order.
__device__ void emit_group_key(const DedupArgs& a, int key, int base) {
  const IndexPtrs& ix = a.ia.ix;
  const int lane = threadIdx.x & 31;
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const int Hkv = a.ia.Hkv, topk = a.ia.topk;
  const int g = key / NB, R = key - g * NB;
  const int o = ixp::seq_of_block(ix.seq, a.ia.B, R);
  const int b = R - ix.seq[o].blk_off;
  const int m = a.d.gsize[R];
  const int32_t* mem = a.d.mlist + a.d.mbeg[R];
  int run = base;
  for (int i0 = 0; i0 < m; i0 += 32) {
    const int i = i0 + lane;
    SeqInfo si{};
    int cnt = 0;
    if (i < m) {
      si = ix.seq[mem[i]];
      cnt = a.d.own_count[(long long)g * NB + si.blk_off + b];
    }
    const int inc = ixp::warp_inclusive_scan(cnt);
    const int my_base = run + inc - cnt;
    const uint32_t* bm = ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words;
    const uint8_t* km = ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq;
    const bool long_row = cnt > 0 && si.words > 2;
    if (cnt > 0 && !long_row) ixp::emit_row_serial(ix, bm, si.words, km, si.q_begin, g, Hkv, topk, my_base);
    unsigned lm = __ballot_sync(0xffffffffu, long_row);
    while (lm) {
      const int l = __ffs(lm) - 1;
      lm &= lm - 1;
      const int l_words = __shfl_sync(0xffffffffu, si.words, l);
      const int l_q0 = __shfl_sync(0xffffffffu, si.q_begin, l);
      const int l_base = __shfl_sync(0xffffffffu, my_base, l);
      const unsigned long long l_bm = __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(bm), l);
      const unsigned long long l_km = __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(km), l);
      ixp::emit_row_warp(ix, reinterpret_cast<const uint32_t*>(l_bm), l_words, reinterpret_cast<const uint8_t*>(l_km),
                         l_q0, g, Hkv, topk, l_base);
    }
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
}

__device__ __forceinline__ long long grid_warp() { return ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; }
__device__ __forceinline__ long long grid_warps() { return ((long long)gridDim.x * blockDim.x) >> 5; }

// scan + emit: the plain build's phase; keys of shared owner blocks are
// queued for the group phase instead of emitted
__device__ void phase_scan_emit_dedup(const DedupArgs& a, unsigned long long* tmp) {
  __shared__ int long_key[kScanTile];
  __shared__ int long_base[kScanTile];
  __shared__ int n_long, n_grp, grp_at;
  __shared__ int2 grp_key[kScanTile];
  const IndexPtrs& ix = a.ia.ix;
  const int B = a.ia.B, Hkv = a.ia.Hkv, topk = a.ia.topk;
  const int n_keys = ix.hdr[kHdrKeys];
  const int NB = ix.hdr[kHdrNB];
  const size_t BMW = (size_t)ix.hdr[kHdrBMW], KMW = (size_t)ix.hdr[kHdrKMW];
  const int warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  unsigned long long pre = 0, all = 0;
  for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
    const unsigned long long v = ix.cta_sums[c];
    all += v;
    if (c < (int)blockIdx.x) pre += v;
  }
  pre = ixp::block_sum(pre, tmp);
  all = ixp::block_sum(all, tmp);
  const unsigned long long kLow = (1ull << 31) - 1;
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    ix.row_ptr[n_keys] = (int)(all >> 31);
    ix.hdr[kHdrNnz] = (int)(all >> 31);
    ix.hdr[kHdrActive] = (int)(all & kLow);
  }
  int lo, hi;
  ixp::key_chunk(n_keys, &lo, &hi);
  unsigned long long carry = pre;
  for (int t0 = lo; t0 < hi; t0 += kScanTile) {
    const int k0 = t0 + threadIdx.x * kScanPerThread;
    int c[kScanPerThread];
    unsigned long long local = 0;
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) {
      c[j] = (k0 + j < hi) ? ix.counts[k0 + j] : 0;
      local += ixp::key_payload(c[j]);
    }
    if (threadIdx.x == 0) {
      n_long = 0;
      n_grp = 0;
    }
    unsigned long long tot;
    unsigned long long run = carry + ixp::block_exclusive_scan(local, tmp, &tot);
    // the member counts of the thread's keys' blocks, read together
    int gs[kScanPerThread];
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) gs[j] = (k0 + j < hi && c[j] > 0) ? a.d.gsize[(k0 + j) % NB] : 0;
    // keys of single-token sequences (one entry each, token 0's): their
    // kmap bytes are read together after the loop
    size_t d_km[kScanPerThread];
    int d_slot[kScanPerThread], d_base[kScanPerThread];
    unsigned deferred = 0;
    // the thread's keys are consecutive: one sequence look-up serves them
    // while their blocks stay in its range
    SeqInfo si{};
    int s_lo = 1, s_hi = 0;
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
          if (r < s_lo || r >= s_hi) {
            si = ix.seq[ixp::seq_of_block(ix.seq, B, r)];
            s_lo = si.blk_off;
            s_hi = si.blk_off + si.nblk;
          }
          const int b = r - si.blk_off;
          const int valid = si.L - 128 * b;
          ix.active_valid[pos] = valid < 128 ? valid : 128;
          if (gs[j] > 1) {
            grp_key[atomicAdd(&n_grp, 1)] = make_int2(key, base);  // queued below, one global add per tile
          } else if (si.tq == 1) {
            d_km[j] = (size_t)g * KMW + (size_t)si.km_off + (size_t)b;
            d_slot[j] = (si.q_begin * Hkv + g) * topk;
            d_base[j] = base;
            deferred |= 1u << j;
          } else if (si.words <= 2) {
            ixp::emit_row_serial(ix, ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words,
                                 si.words, ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq,
                                 si.q_begin, g, Hkv, topk, base);
          } else {
            const int at = atomicAdd(&n_long, 1);
            long_key[at] = key;
            long_base[at] = base;
          }
        }
      }
      run += ixp::key_payload(c[j]);
    }
    int d_k[kScanPerThread];
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) d_k[j] = (deferred >> j) & 1u ? ix.kmap[d_km[j]] : 0;
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) {
      if ((deferred >> j) & 1u) {
        const int slot = d_slot[j] + d_k[j];
        ix.entries[d_base[j]] = slot;
        ix.slot_entry[slot] = d_base[j];
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && n_grp > 0) grp_at = atomicAdd(&ix.hdr[kHdrGroupKeys], n_grp);
    __syncthreads();
    for (int i = threadIdx.x; i < n_grp; i += blockDim.x) a.d.gkeys[grp_at + i] = grp_key[i];
    for (int i = warp; i < n_long; i += n_warps) {
      const int key = long_key[i];
      const int g = key / NB, r = key - g * NB;
      const SeqInfo si = ix.seq[ixp::seq_of_block(ix.seq, B, r)];
      const int b = r - si.blk_off;
      ixp::emit_row_warp(ix, ix.bitmap + (size_t)g * BMW + (size_t)si.bm_off + (size_t)b * si.words, si.words,
                         ix.kmap + (size_t)g * KMW + (size_t)si.km_off + (size_t)b * si.tq, si.q_begin, g, Hkv,
                         topk, long_base[i]);
    }
    __syncthreads();
    carry += tot;
  }
}

// Four CTAs per SM (64 registers): the phases are chains of dependent
// reads, and twice the warps of the other index kernels keep twice the reads
// in flight.
constexpr int kDedupCtasPerSm = 3;
__global__ void __launch_bounds__(kIndexThreads, kDedupCtasPerSm) k_index_dedup(DedupArgs a) {
  __shared__ unsigned long long tmp[3 * 33];
  __shared__ int32_t rowbuf[ixp::kMarkWarps][256];
  const IndexPtrs& ix = a.ia.ix;
  int* bar = ix.hdr + kHdrBarCount;
  int epoch = 0;
  int* flags = ix.hdr + kHdrFlags;
  const unsigned nb = gridDim.x;
  if (blockIdx.x == 0) {
    ixp::phase_seq(ix, a.ia.cu, a.ia.lens, a.ia.B, a.ia.total_q, a.ia.Hkv, a.ia.cap_len, a.ia.causal,
                   reinterpret_cast<long long*>(tmp));
    if (threadIdx.x == 0) ix.hdr[kHdrDedup] = 1;
  }
  ixp::phase_token_seq(ix, a.ia.cu, a.ia.B, a.ia.total_q);
  for (long long p = grid_tid(); p < a.num_pages; p += grid_threads()) a.d.page_min[p] = ~0ull;
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  ixp::phase_zero(ix, a.ia.Hkv, ixp::SeqTotals{ix.hdr[kHdrNB], ix.hdr[kHdrBMW], ix.hdr[kHdrKMW]});
  phase_offer(a);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  ixp::phase_mark(ix, a.ia.sel, a.ia.total_q, a.ia.Hkv, a.ia.topk, a.ia.causal, rowbuf, false);
  phase_owner(a);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  phase_fold(a);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  ixp::phase_key_reduce(ix, tmp);
  for (long long i = grid_warp(); i < ix.hdr[kHdrGroups]; i += grid_warps()) walk_members(a, a.d.glist[i]);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  phase_scan_emit_dedup(a, tmp);
  if (!grid_barrier(bar, flags, nb, epoch)) return;
  for (long long i = grid_warp(); i < ix.hdr[kHdrGroupKeys]; i += grid_warps()) {
    const int2 gk = a.d.gkeys[i];
    emit_group_key(a, gk.x, gk.y);
  }
}

}  // namespace


cudaError_t launch_build_index_dedup(const mxsa_problem& p, const int32_t* sel, const int64_t* cu,
                                     const int32_t* lens, const int32_t* block_tables, const IndexPtrs& ix,
                                     const DedupPtrs& d, cudaStream_t st) {
  DedupArgs a;
  a.ia = ixp::IndexArgs{ix, sel, cu, lens, p.num_seqs, p.total_q, p.num_kv_heads, p.topk,
                        p.max_pages_per_seq * p.page_size, p.causal};
  a.d = d;
  a.bt = block_tables;
  a.max_pages = p.max_pages_per_seq;
  a.num_pages = p.num_pages;
  a.ps = p.page_size;
  const int grid = coop_grid(reinterpret_cast<const void*>(k_index_dedup), kIndexThreads, kDedupCtasPerSm);
  if (grid <= 0) return cudaErrorNotSupported;
  cudaError_t e = cudaMemsetAsync(ix.hdr, 0, kHdrInts * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_index_dedup), dim3(grid), dim3(kIndexThreads),
                                     args, 0, st);
}

}  // namespace mxsa
