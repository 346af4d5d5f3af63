// KV-outer forward for KV-stationary work items (fw-ai/minimax-kernels
// README, intro: "loads a selected KV block once and processes all queries
// that selected it").  A work item is up to 4 tiles of 128 (entry, head)
// rows of one key (kv head, sequence, block): the block's K and V pages are
// TMA-loaded once per item and every tile of rows is multiplied against them.
//
// Persistent kernel, one CTA per SM, 352 threads (this phase's roles):
//   warps 0-3, 4-7  two softmax warpgroups; the CTA's tiles alternate
//              between them (tile j -> warpgroup j % 2) so that one group's
//              softmax overlaps the other group's MMAs, loads and stores.
//              Per tile a group brings the tile's q rows into its buffer
//              (TMA boxes, or a warp gather when G is not a multiple of 8),
//              turns S = q k^T (TMEM) into P = exp(S - m), written back to
//              TMEM over S as the p v operand, and after O = P v writes
//              o = O / l and lse per row straight from TMEM.  Row r of a tile is
//              thread r of its group and TMEM lane r.  For FP8 and NVFP4
//              caches warpgroup n % 2 widens the CTA's n-th block to
//              BF16/FP16 in the stage (exactly), whether or not it owns a
//              tile of that item.
//   warp 8     producer: decodes items (key -> kv head, sequence, block),
//              walks the block table and TMA-loads the block's K and V pages
//              into a double-buffered stage (FP8: e4m3 rows into the
//              stage's V half, widened in place; NVFP4: into a staging
//              tile).
//   warps 9, 10  MMA issuers, one per softmax group (tcgen05.mma,
//              cta_group::1, M = N = 128, K = 16 per instruction, FP32
//              accumulate in TMEM: S and O of each group, 512 columns owned
//              by warp 9): q k^T then p v of each of the group's tiles.
//
// Shared-memory operands use the 128-byte swizzled K-major layout (q, K)
// and the 128-byte swizzled MN-major layout (V as the B operand of P V);
// P is the TMEM (A) operand of P V.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "fwd_decode.cuh"

namespace mxsa {

namespace {

constexpr int kThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTileBytes = 32768;  // 128 rows x 128 x 16-bit
constexpr uint32_t kStageBytes = 2 * kTileBytes;

struct ItemInfo {
  int32_t g, s, b, valid, e0, n, L, tq, q_begin, pad0, pad1, pad2, pad3, pad4, pad5, pad6;
};

constexpr int kMaxItemEntries = MXSA_ITEM_TILES * (MXSA_TILE_ROWS / 8);

struct Ctrl {
  // stg_full[n % 2]: item n staged.  One barrier per widening group, so
  // that each group waits for every phase of its own barrier in order.
  uint64_t kv_full[2], kv_empty[2], stg_full[2], stg_empty, q_full[2], s_full[2], p_full[2], o_full[2], done;
  uint64_t epi_turn[2];  // epi_turn[g]: the other group finished an epilogue
  uint32_t tmem_base;
  int32_t abort_flag;
  ItemInfo info[2];
  // the tokens of each stage's item entries when q comes by TMA (G >= 8:
  // at most 4 tiles x 16 entries)
  int32_t tok[2][kMaxItemEntries];
};

struct FwdArgs {
  const uint8_t* q;
  const int32_t* block_tables;
  const SeqInfo* seq;
  const int32_t* token_seq;
  const int32_t* entries;
  const int4* items;
  const int32_t* cta_ptr;
  const int32_t* idx_hdr;
  const int32_t* sch_hdr;
  void* part_o;  // partial rows: FP32 when part32, else the 16-bit q dtype
  float* part_lse;
  int32_t* flags;
  int32_t num_seqs, Hq, Hkv, G, topk, page_size, max_pages, num_pages, causal, kv_fp8, ab_bf16, per_tile;
  int32_t part32;
  int32_t kv_fp4;     // NVFP4 (kv_fp8 is set too: staged and widened); scale rows from kbase / vbase
  const uint8_t* kbase;
  const uint8_t* vbase;
  int32_t q_tma;      // q rows of a tile come by TMA (G % 8 == 0; the map tmqs exists)
  int32_t* claim;     // schedule header word: next item to claim
  int32_t* sch_hdr_mut;  // the schedule header (claim and exit counters)
  float scale_log2;
};

// smem offsets from the 1024-aligned base
constexpr uint32_t kOffKV = 0;                            // 2 stages x (K, V)
constexpr uint32_t kOffQP = 2 * kStageBytes;              // 2 groups x q tile
constexpr uint32_t kOffStg = kOffQP + 2 * kTileBytes;     // NVFP4 staging (K, V code and scale rows), 32 KB
constexpr uint32_t kCtrlBf16 = kOffStg;
constexpr uint32_t kCtrlFp8 = kOffStg + kTileBytes;  // widened caches (FP8 widens in place and leaves the staging tile unused)

__device__ __forceinline__ int seq_of_block(const SeqInfo* seq, int B, int r) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq[mid].blk_off <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk16) {
  // byte offset of 16-byte chunk `chunk16` (0..15) of row `row` in a
  // [128 rows][128 x 16-bit] tile stored as two 128B-swizzled halves
  return (chunk16 >> 3) * 16384u + row * 128u + (((chunk16 & 7u) ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// two e4m3 bytes (low byte first) -> two 16-bit values of the MMA dtype
__device__ __forceinline__ uint32_t widen_e4m3x2(uint16_t v, int bf16) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  if (!bf16) return h2;
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(h);  // exact
  return pack2(f.x, f.y, 1);     // exact: e4m3 values are representable in bf16
}

// The tile entry whose q boxes lane `wl` of warp `w` (0..3) of a softmax
// group issues: warp w holds tile rows 32w .. 32w + 31, and an entry's G rows
// start at row e * G, so its entries are those starting in that range (for
// G > 32 some warps have none).  A value past the tile's entries means none.
__device__ __forceinline__ int qbox_entry(int w, int wl, int G) {
  const int first = (32 * w + G - 1) / G, last = (32 * w + 32 + G - 1) / G;  // [first, last)
  return first + wl < last ? first + wl : 1 << 30;
}

// A wait's outcome made uniform across the warp (the TMEM loads and stores
// that follow are warp-collective).  The warps of a softmax group do not
// wait for one another: every hand-off between them and the other roles is
// an mbarrier, and a wait that gives up raises the CTA's abort flag, which
// ends every other wait.
__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// Per-row state a group keeps from a tile's softmax to its epilogue.  The
// rows of a tile are consecutive partial rows: row r is orow0 + r.
struct RowState {
  size_t orow0;
  float m2, l;
  int rows;  // rows of the tile that hold an (entry, head) pair
};

// P = exp2(S * scale_log2 - m2) of one row over 64 of the block's keys
// (half h: keys 64h .. 64h + 63, S values in sv), packed in pairs to the MMA
// operand type and written to TMEM columns tP + 32h .. + 31 of the row's
// lane (over S columns already read); returns the partial row sum.
// kFull: every key is visible (no length or causal limit).
template <bool kBf16, bool kFull>
__device__ __forceinline__ float softmax_store_p(const float* sv, int h, float scale_log2, float m2, int lim,
                                                 uint32_t tP) {
  float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
  uint32_t pk[32];
#pragma unroll
  for (int cl = 0; cl < 8; ++cl) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int kl = cl * 8 + 2 * i, k0 = 64 * h + kl;
      float p0 = ex2_approx(fmaf(sv[kl], scale_log2, -m2));
      float p1 = ex2_approx(fmaf(sv[kl + 1], scale_log2, -m2));
      if (!kFull) {
        p0 = k0 < lim ? p0 : 0.f;
        p1 = k0 + 1 < lim ? p1 : 0.f;
      }
      if (i == 0) l0 += p0 + p1;
      if (i == 1) l1 += p0 + p1;
      if (i == 2) l2 += p0 + p1;
      if (i == 3) l3 += p0 + p1;
      if (kBf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        pk[4 * cl + i] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __half2 h = __floats2half2_rn(p0, p1);
        pk[4 * cl + i] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
  }
  tmem_st32(tP + 32 * h, pk);
  return (l0 + l1) + (l2 + l3);
}

// Runs the CTA's KV-stationary items (all kThreads threads; 1024-aligned
// shared memory `sm`; TMEM base `tmem` with 512 columns).  kKV: the cache
// kind (kKv16, kKvFp8, kKvFp4); widened caches write FP32 partial rows,
// 16-bit ones rows in the q dtype.
template <int kKV>
__device__ __forceinline__ void kv_stationary_body(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                                   const CUtensorMap& tmqs, const FwdArgs& a, uint8_t* sm,
                                                   uint32_t tmem) {
  constexpr bool kPart32 = kind_partials_fp32(kKV);
  Ctrl& c = *reinterpret_cast<Ctrl*>(sm + (a.kv_fp8 ? kCtrlFp8 : kCtrlBf16));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Items are claimed dynamically (a global counter), in item order, by the
  // producer, which publishes each one in its stage's info and ends with an
  // item of no entries; every role follows that sequence.
  const int n_items = a.sch_hdr[kSchItems];
  if (n_items <= 0) return;  // uniform: nothing to do

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c.kv_full[i], a.kv_fp8 ? 128 : 1);  // FP8: the widening group arrives
      // a stage is refilled after both MMA issuers committed it and every
      // softmax thread read its info (so no role lags two phases behind)
      mbar_init(&c.kv_empty[i], 2 + 256);
      mbar_init(&c.q_full[i], a.q_tma ? 1 : 128);  // TMA: one arrival plus the bytes
      mbar_init(&c.s_full[i], 1);
      mbar_init(&c.p_full[i], 128);
      mbar_init(&c.o_full[i], 1);
      mbar_init(&c.stg_full[i], 1);
    }
    mbar_init(&c.epi_turn[0], 128);
    mbar_init(&c.epi_turn[1], 128);
    mbar_init(&c.stg_empty, 128);
    mbar_init(&c.done, 2);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &c.abort_flag;
  const uint32_t sbase = smem_u32(sm);
  const int per_tile = a.per_tile;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Lane 0 claims, decodes and loads the items; on the TMA q path the warp
    // first copies the item's entry tokens next to its info, so that the
    // softmax groups read them from shared memory.
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      if (a.q_tma) tma_prefetch_desc(&tmqs);
    }
    const int NB = a.idx_hdr[kHdrNB];
    const int ps = a.page_size;
    const int npg = ps == 128 ? 1 : 2;
    const int tok_div = a.Hkv * a.topk;
    int n = 0;
    bool ok = true, ended = false;
    int it = 0;
    if (lane == 0) it = atomicAdd(a.claim, 1);
    it = __shfl_sync(0xffffffffu, it, 0);
    for (; ok; ++n) {
      const int st = n & 1, use = n >> 1;
      if (lane == 0)
        ok = mbar_wait(&c.kv_empty[st], (use & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (it >= n_items) {  // no item left: publish the end
        if (lane == 0) {
          ItemInfo end{};
          c.info[st] = end;
          mbar_arrive(a.kv_fp8 ? &c.stg_full[st] : &c.kv_full[st]);
        }
        ended = true;
        break;
      }
      int next = 0;
      if (lane == 0) next = atomicAdd(a.claim, 1);  // claimed one item ahead: its latency overlaps this item
      const int4 itm = a.items[it];
      if (a.q_tma) {
        const int ne = min(itm.z, kMaxItemEntries);
        for (int e = lane; e < ne; e += 32) c.tok[st][e] = __ldg(a.entries + itm.y + e) / tok_div;
      }
      __syncwarp();  // the tokens are written before lane 0 publishes the item
      if (lane == 0) {
        const int key = itm.x;
        const int g = key / NB, r = key - g * NB;
        const int s = seq_of_block(a.seq, a.num_seqs, r);
        const SeqInfo si = a.seq[s];
        const int b = r - si.blk_off;
        const int valid = min(128, si.L - 128 * b);
        // physical pages of the block (1 for 128-token pages, 1-2 for 64)
        int pages[2] = {-1, -1};
        for (int pg = 0; pg < npg; ++pg) {
          if (pg * 64 >= valid) continue;
          const int lp = ps == 128 ? b : 2 * b + pg;
          const int phys = a.block_tables[(size_t)s * a.max_pages + lp];
          if (phys < 0 || phys >= a.num_pages) {
            atomicOr(a.flags, MXSA_FLAG_PAGE);
            continue;
          }
          pages[pg] = phys;
        }
        ItemInfo inf;
        inf.g = g; inf.s = s; inf.b = b; inf.valid = valid; inf.e0 = itm.y; inf.n = itm.z;
        inf.L = si.L; inf.tq = si.tq; inf.q_begin = si.q_begin;
        c.info[st] = inf;
        const int present = (pages[0] >= 0) + (pages[1] >= 0);
        if (!a.kv_fp8) {
          uint8_t* kdst = sm + kOffKV + st * kStageBytes;
          uint8_t* vdst = kdst + kTileBytes;
          mbar_arrive_expect_tx(&c.kv_full[st], (uint32_t)present * (uint32_t)ps * 512u);
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            const int z = pages[pg] * a.Hkv + g;
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(kdst + h * 16384 + pg * 8192, &tmk, &c.kv_full[st], h * 64, 0, z);
              tma_load_3d(vdst + h * 16384 + pg * 8192, &tmv, &c.kv_full[st], h * 64, 0, z);
            }
          }
        } else if (!a.kv_fp4) {
          // FP8: the e4m3 rows land in the stage's V half (K rows at 0, V
          // rows at 16 KB, 128 bytes each), where the widening group widens
          // them in place
          uint8_t* vhalf = sm + kOffKV + st * kStageBytes + kTileBytes;
          uint64_t* sf = &c.stg_full[st];
          mbar_arrive_expect_tx(sf, (uint32_t)present * (uint32_t)ps * 256u);
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            const int z = pages[pg] * a.Hkv + g;
            tma_load_3d(vhalf + pg * 8192, &tmk, sf, 0, 0, z);
            tma_load_3d(vhalf + 16384 + pg * 8192, &tmv, sf, 0, 0, z);
          }
        } else {
          // NVFP4: into the staging tile once the previous block was widened
          // out of it (stg_empty): code rows by TMA, scale rows by bulk copy
          // (K at 0, V at 16 KB of the staging tile; codes, then scales at
          // 8 KB); the widening group fills the stage
          ok = mbar_wait(&c.stg_empty, (n & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (ok) {
            uint8_t* stg = sm + kOffStg;
            uint64_t* sf = &c.stg_full[st];
            mbar_arrive_expect_tx(sf, (uint32_t)present * (uint32_t)ps * 144u);
            for (int pg = 0; pg < npg; ++pg) {
              if (pages[pg] < 0) continue;
              const int z = pages[pg] * a.Hkv + g;
              const size_t so = (size_t)z * ps * 72 + (size_t)ps * 64;
              tma_load_3d(stg + pg * ps * 64, &tmk, sf, 0, 0, z);
              tma_load_3d(stg + 16384 + pg * ps * 64, &tmv, sf, 0, 0, z);
              bulk_load(stg + 8192 + pg * ps * 8, a.kbase + so, (uint32_t)ps * 8u, sf);
              bulk_load(stg + 16384 + 8192 + pg * ps * 8, a.vbase + so, (uint32_t)ps * 8u, sf);
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;  // NVFP4 staging gave up: item n issued no loads
      it = __shfl_sync(0xffffffffu, next, 0);
    }
    // drain: every load lane 0 issued has landed before the CTA may exit.
    // After the end item (published on stage n % 2) item n - 2 has landed
    // for sure (its stage was released for the end item), and its barrier
    // has moved on, so only item n - 1 is waited for.  NVFP4: staging item
    // n - 1 needed item n - 2 widened, so only n - 1.
    if (lane == 0) {
      const int k0 = (ended || a.kv_fp4) ? n - 1 : n - 2;
      for (int k = std::max(0, k0); k < n; ++k)
        mbar_drain(a.kv_fp8 ? &c.stg_full[k & 1] : &c.kv_full[k & 1], (k >> 1) & 1, a.flags, MXSA_FLAG_TIMEOUT,
                   kWaitLimitNs);
    }
  } else if (warp >= kMmaWarp) {
    // ---------------------------------------------------------- MMA issuers
    // Warp 9 + g (lane 0) issues the MMAs of softmax group g (its tiles
    // j = g, g + 2, ...): q k^T once the tile's q rows are in and the
    // group's previous p v is done (P is kept in TMEM over S), then p v,
    // with P as the TMEM operand, once the group wrote P.
    // Each issuer waits only on its own group, so one group's MMAs never
    // queue behind the other group's inputs; a stage is released after both
    // issuers committed it (kv_empty counts two arrivals).
    if (lane == 0) {
      const int g = warp - kMmaWarp;
      const uint32_t id_qk = idesc_f16(128, 128, (uint32_t)a.ab_bf16, 0, 0);
      const uint32_t id_pv = idesc_f16(128, 128, (uint32_t)a.ab_bf16, 0, 1);
      const uint32_t q_s = sbase + kOffQP + g * kTileBytes;  // q rows of group g
      const uint32_t tS = tmem + g * 256, tO = tS + 128;
      int n = 0, j = 0, jprev = -1;
      bool ok = true;
      for (; ok; ++n) {
        const int st = n & 1, use = n >> 1;
        ok = mbar_wait(&c.kv_full[st], use & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        const int n_entries = c.info[st].n;
        if (n_entries == 0) break;  // the end
        const int ntiles = (n_entries + per_tile - 1) / per_tile;
        const uint32_t k_s = sbase + kOffKV + st * kStageBytes, v_s = k_s + kTileBytes;
        for (int t = 0; t < ntiles && ok; ++t, ++j) {
          if ((j & 1) != g) continue;
          ok = mbar_wait(&c.q_full[g], (j >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (!ok) break;
          if (jprev >= 0) {  // S is overwritten only after the previous p v read P
            ok = mbar_wait(&c.o_full[g], (jprev >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
            mma_f16_ss(tS, smem_desc_sw128(q_s + off, 0, 1024), smem_desc_sw128(k_s + off, 0, 1024), id_qk, ks > 0);
          }
          mma_commit(&c.s_full[g]);
          ok = mbar_wait(&c.p_full[g], (j >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ts(tO, tS + ks * 8, smem_desc_sw128(v_s + ks * 2048u, 16384, 1024), id_pv, ks > 0);
          mma_commit(&c.o_full[g]);
          jprev = j;
        }
        if (ok) mma_commit(&c.kv_empty[st]);  // this issuer's share of the stage is done
      }
      // drain: all MMAs of both issuers complete before TMEM is freed (done
      // counts two arrivals)
      mma_commit(&c.done);
      mbar_drain(&c.done, 0, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------ softmax groups
    const int grp = warp >> 2;     // 0 or 1
    const int r = tid & 127;       // tile row == TMEM lane
    // With the dedup index a key's rows may come from several sequences
    // (the same physical block at the same logical position): each row then
    // takes its causal position from its own token's sequence.
    const bool row_seq = a.causal && a.idx_hdr[kHdrDedup] != 0;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + grp * 256 + lane_addr, tO = tS + 128;
    const uint32_t qp = sbase + kOffQP + grp * kTileBytes;
    const int bf16 = a.ab_bf16;
    int n = 0, j = 0;
    bool ok = true;
    const int wl = tid & 31, wrow0 = (warp & 3) * 32;  // lane; the warp's first tile row
    RowState pend{0, -INFINITY, 0.f, 0};
    int pend_j = -1;
    int jq = -1;  // the group's last tile whose q rows were requested by TMA
    // epilogue of this group's previous tile: o = O / l, lse = (m2 + log2 l)
    // ln 2.  O is read in the 16x256b shape, in which four consecutive lanes
    // hold 8 consecutive columns of one row (two per lane).  FP32 partials:
    // each lane stores its two values, so each store instruction writes
    // eight whole 32-byte sectors (8 rows x 8 columns).  16-bit partials:
    // after packing, one exchange between lane pairs leaves each lane 4
    // consecutive values of one of two adjacent 8-column chunks, so each
    // store instruction again writes eight whole sectors (8 rows x 16
    // columns).  Both straight from registers; the epilogue runs while the
    // next tile's q k^T is in flight.
    // The groups take turns at the epilogue, in tile order (tile j's after
    // tile j - 1's), so that one group's stores run while the other group
    // computes instead of both groups storing at once at half the rate.
    int n_epi = 0;  // epilogues this group has run
    auto epilogue = [&]() -> bool {
      // this group's epilogue m is tile 2m + grp; it follows tile 2m + grp - 1
      const int m = n_epi;
      if (grp == 1 || m > 0) {
        const int ph = grp == 1 ? m : m - 1;  // the other group's epilogue it waits for
        if (!warp_all(mbar_wait(&c.epi_turn[grp], ph & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs)))
          return false;
      }
      const float inv_l = pend.l > 0.f ? 1.f / pend.l : 0.f;
      if (kPart32 && wrow0 < pend.rows) {  // a warp of padding rows has nothing to store
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int ra = hh * 16 + (wl >> 2), rb = ra + 8;  // the warp's rows this lane stores
          const float sa = __shfl_sync(0xffffffffu, inv_l, ra), sb = __shfl_sync(0xffffffffu, inv_l, rb);
          const bool oka = wrow0 + ra < pend.rows, okb = wrow0 + rb < pend.rows;
          float* ga = static_cast<float*>(a.part_o) + (pend.orow0 + wrow0 + ra) * 128 + 2 * (wl & 3);
          float* gb = ga + 8 * 128;
          float v0[32], v1[32];
          tmem_ld16x256b_x8(tO + ((uint32_t)(hh * 16) << 16), v0);
          tmem_ld16x256b_x8(tO + ((uint32_t)(hh * 16) << 16) + 64, v1);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (oka) st_global_cs_v2f(ga + 8 * c, v0[4 * c] * sa, v0[4 * c + 1] * sa);
            if (okb) st_global_cs_v2f(gb + 8 * c, v0[4 * c + 2] * sb, v0[4 * c + 3] * sb);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (oka) st_global_cs_v2f(ga + 64 + 8 * c, v1[4 * c] * sa, v1[4 * c + 1] * sa);
            if (okb) st_global_cs_v2f(gb + 64 + 8 * c, v1[4 * c + 2] * sb, v1[4 * c + 3] * sb);
          }
        }
      } else if (!kPart32 && wrow0 < pend.rows) {
        const int qd = wl & 3, odd = wl & 1;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int ra = hh * 16 + (wl >> 2), rb = ra + 8;  // the warp's rows this lane stores
          const float sa = __shfl_sync(0xffffffffu, inv_l, ra), sb = __shfl_sync(0xffffffffu, inv_l, rb);
          const bool oka = wrow0 + ra < pend.rows, okb = wrow0 + rb < pend.rows;
          uint16_t* ga = static_cast<uint16_t*>(a.part_o) + (pend.orow0 + wrow0 + ra) * 128;
          uint16_t* gb = ga + 8 * 128;
          float vv[2][32];
          tmem_ld16x256b_x8(tO + ((uint32_t)(hh * 16) << 16), vv[0]);
          tmem_ld16x256b_x8(tO + ((uint32_t)(hh * 16) << 16) + 64, vv[1]);
          tmem_ld_wait();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const float* v = vv[half];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              // chunks c0 = 2u, c1 = 2u + 1: this lane holds columns 8c + 2qd, +1
              // of each; an even lane keeps chunk c0 and takes its odd
              // neighbour's part of it, an odd lane keeps c1 and takes its even
              // neighbour's part of c1
              const int c0 = 2 * u, c1 = 2 * u + 1;
              const uint32_t a0 = pack2(v[4 * c0] * sa, v[4 * c0 + 1] * sa, bf16);
              const uint32_t a1 = pack2(v[4 * c1] * sa, v[4 * c1 + 1] * sa, bf16);
              const uint32_t b0 = pack2(v[4 * c0 + 2] * sb, v[4 * c0 + 3] * sb, bf16);
              const uint32_t b1 = pack2(v[4 * c1 + 2] * sb, v[4 * c1 + 3] * sb, bf16);
              const uint32_t ra_x = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
              const uint32_t rb_x = __shfl_xor_sync(0xffffffffu, odd ? b0 : b1, 1);
              const int col = 64 * half + (odd ? 8 * c1 + 2 * qd - 2 : 8 * c0 + 2 * qd);
              if (oka) st_global_cs_v2u(ga + col, odd ? ra_x : a0, odd ? a1 : ra_x);
              if (okb) st_global_cs_v2u(gb + col, odd ? rb_x : b0, odd ? b1 : rb_x);
            }
          }
        }
      }
      if (r < pend.rows)
        __stcs(&a.part_lse[pend.orow0 + r],
               pend.l > 0.f ? (pend.m2 + lg2_approx(pend.l)) * 0.69314718055994530942f : -INFINITY);
      tc_fence_before();
      mbar_arrive(&c.epi_turn[grp ^ 1]);  // the other group's turn
      ++n_epi;
      return true;
    };
    for (; ok; ++n) {
      const int st = n & 1, use = n >> 1;
      if (kKV != dec::kKv16 && st == grp) {
        // widen the staged block (row r of K and V) into the stage; rows
        // past the valid tokens become zero.  The producer loaded this block
        // only after kv_empty of the stage, so the stage is free.
        ok = warp_all(mbar_wait(&c.stg_full[st], use & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        const int valid = c.info[st].n > 0 ? c.info[st].valid : 0;  // the end item stages nothing
        for (int kv = 0; kv < 2 && kKV == dec::kKvFp4; ++kv) {
          const uint32_t stg = sbase + kOffStg;
          const uint32_t dst = sbase + kOffKV + st * kStageBytes + kv * kTileBytes;
          if (r < valid)
            dec::widen_fp4_row(stg + kv * 16384 + r * 64, stg + kv * 16384 + 8192 + r * 8, dst, r, bf16);
          else
            for (int ch = 0; ch < 16; ++ch) st_shared_v4(dst + swz(r, ch), 0, 0, 0, 0);
        }
        // FP8, in place: the e4m3 rows sit in the stage's V half (K row r at
        // r * 128, V row r at 16 KB + r * 128).  K widens into the K half.
        // Widened V row r covers bytes r * 128 of both 16 KB halves of the V
        // half: e4m3 K row r (already widened) and e4m3 V row r, which this
        // thread reads whole before writing, so no thread touches another
        // thread's row.
        for (int kv = 0; kv < 2 && kKV == dec::kKvFp8; ++kv) {
          const uint32_t src = sbase + kOffKV + st * kStageBytes + kTileBytes + kv * 16384 + r * 128;
          const uint32_t dst = sbase + kOffKV + st * kStageBytes + kv * kTileBytes;
          uint4 raw[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const int c8 = (cc + r) & 7;  // rotate to spread banks
            raw[cc] = r < valid ? ld_shared_v4(src + c8 * 16) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const int c8 = (cc + r) & 7;
            const uint32_t w4[4] = {raw[cc].x, raw[cc].y, raw[cc].z, raw[cc].w};
            uint32_t o8[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o8[2 * i] = widen_e4m3x2((uint16_t)(w4[i] & 0xffffu), bf16);
              o8[2 * i + 1] = widen_e4m3x2((uint16_t)(w4[i] >> 16), bf16);
            }
            st_shared_v4(dst + swz(r, 2 * c8), o8[0], o8[1], o8[2], o8[3]);
            st_shared_v4(dst + swz(r, 2 * c8 + 1), o8[4], o8[5], o8[6], o8[7]);
          }
        }
        fence_proxy_async_smem();
        if (kKV == dec::kKvFp4 && c.info[st].n > 0) mbar_arrive(&c.stg_empty);
        mbar_arrive(&c.kv_full[st]);
      }
      // every group reads every item's info (the tile count decides the
      // groups' alternation), then lets the stage go
      ok = warp_all(mbar_wait(&c.kv_full[st], use & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
      if (!ok) break;
      const ItemInfo inf = c.info[st];
      if (inf.n == 0) break;  // the end
      const int ntiles = (inf.n + per_tile - 1) / per_tile;
      // TMA q path: the tokens this thread needs for the group's tiles of
      // the item (at most two: an item has at most 4 tiles), taken from the
      // producer's copy before the stage is let go: row r's (for its key
      // limit) and the entry whose q boxes this lane issues
      const int qe = qbox_entry(warp & 3, wl, a.G);
      int tk_row0 = -1, tk_row1 = -1, tk_box0 = 0, tk_box1 = 0;
      if (a.q_tma) {
        const int t0 = (j & 1) == grp ? 0 : 1;  // the group's first tile of the item
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int t = t0 + 2 * i;
          if (t >= ntiles) break;
          const int ne = min(per_tile, inf.n - t * per_tile);
          const int tr = r < ne * a.G ? c.tok[st][t * per_tile + r / a.G] : -1;
          const int tb = qe < ne ? c.tok[st][t * per_tile + qe] : 0;
          if (i == 0) { tk_row0 = tr; tk_box0 = tb; } else { tk_row1 = tr; tk_box1 = tb; }
        }
      }
      mbar_arrive(&c.kv_empty[st]);  // this thread read the info and tokens
      bool first = true;  // this group's first tile of the item
      for (int t = 0; t < ntiles && ok; ++t, ++j) {
        if ((j & 1) != grp) continue;
        const int et0 = inf.e0 + t * per_tile;
        const int ne = min(per_tile, inf.n - t * per_tile);
        const int rows = ne * a.G;
        // row r's token (-1: padding row), which gives its q row and key
        // limit: from the copy above, or (warp gather path) the entry list
        int tok = (t >> 1) ? tk_row1 : tk_row0;
        if (!a.q_tma) tok = r < rows ? __ldg(a.entries + et0 + r / a.G) / (a.Hkv * a.topk) : -1;
        // the token's causal position (loaded here, used after the epilogue)
        int pos = 0;
        if (tok >= 0) {
          if (row_seq) {
            const SeqInfo* ts = a.seq + __ldg(a.token_seq + tok);
            pos = __ldg(&ts->L) - __ldg(&ts->tq) + (tok - __ldg(&ts->q_begin));
          } else {
            pos = inf.L - inf.tq + (tok - inf.q_begin);
          }
        }
        // ---- this tile's q rows into the group's buffer, free since the
        // group's previous q k^T completed (it waited for that S)
        if (a.q_tma) {
          // by TMA: an entry's G rows (its token, this kv head's q heads) are
          // consecutive q rows, one box per 64-column half, landing at whole
          // 1024-byte swizzle atoms (G is a multiple of 8).  The warp holding
          // an entry's first row issues its boxes, so the four warps share
          // the issue.  Rows past the tile's entries keep stale values: their
          // rows of S, P and O are never stored.
          if (r == 0) mbar_arrive_expect_tx(&c.q_full[grp], (uint32_t)rows * 256u);
          if (qe < ne) {
            uint8_t* dst = sm + kOffQP + grp * kTileBytes + qe * a.G * 128;
            const int row0 = ((t >> 1) ? tk_box1 : tk_box0) * a.Hq + inf.g * a.G;
            tma_load_2d(dst, &tmqs, &c.q_full[grp], 0, row0);
            tma_load_2d(dst + 16384, &tmqs, &c.q_full[grp], 64, row0);
          }
          jq = j;
        } else {
          const int qrow = tok >= 0 ? tok * a.Hq + inf.g * a.G + r % a.G : -1;
          // coalesced gather: in round i the two half-warps read whole
          // 256-byte q rows (the warp's rows 2i and 2i + 1, one 16-byte chunk
          // per lane)
          uint4 v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int src_row = __shfl_sync(0xffffffffu, qrow, 2 * i + (wl >> 4));
            v[i] = src_row >= 0 ? __ldg(reinterpret_cast<const uint4*>(a.q + (size_t)src_row * 256) + (wl & 15))
                                : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_shared_v4(qp + swz(wrow0 + 2 * i + (wl >> 4), wl & 15), v[i].x, v[i].y, v[i].z, v[i].w);
          fence_proxy_async_smem();
          mbar_arrive(&c.q_full[grp]);
        }
        if (pend_j >= 0) {
          // the previous tile's O is complete once its p v is done
          ok = warp_all(mbar_wait(&c.o_full[grp], (pend_j >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT,
                                   kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          ok = epilogue();
          if (!ok) break;
        }
        int lim = 0;
        if (tok >= 0) {
          lim = inf.valid;
          if (a.causal) lim = min(lim, pos - 128 * inf.b + 1);
        }
        if (first && kKV == dec::kKv16 && r >= inf.valid) {
          // keys past the sequence end must not bring stale values (they may
          // be NaN bit patterns) into P V.  Both groups zero the rows before
          // their own first p v of the item (the fence before p_full orders
          // the stores): zeros written twice are harmless, and neither
          // group's p v then depends on the other's progress.
          const uint32_t vs = sbase + kOffKV + st * kStageBytes + kTileBytes;
          for (int ch = 0; ch < 16; ++ch) st_shared_v4(vs + swz(r, ch), 0, 0, 0, 0);
        }
        first = false;
        // ---- softmax of the row
        ok = warp_all(mbar_wait(&c.s_full[grp], (j >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        float m2 = -INFINITY, l = 0.f;
        {
          // S is read from TMEM twice, 64 columns at a time (the maximum, then
          // P), so that only 64 scores are live; four independent maxima and
          // sums keep the dependency chains short
          const bool full = __all_sync(0xffffffffu, lim >= 128);
          // padding rows' P is never used (their output rows are not stored),
          // so a warp of padding rows skips the softmax
          const bool dead = wrow0 >= rows;
          float m0 = -INFINITY, m1 = -INFINITY, m3 = -INFINITY, m4 = -INFINITY;
#pragma unroll
          for (int h = 0; h < 2 && !dead; ++h) {
            float sv[64];
            tmem_ld32(tS + h * 64, sv);
            tmem_ld32(tS + h * 64 + 32, sv + 32);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 64; k += 4) {
              const int kk = 64 * h + k;
              m0 = fmaxf(m0, full || kk < lim ? sv[k] : -INFINITY);
              m1 = fmaxf(m1, full || kk + 1 < lim ? sv[k + 1] : -INFINITY);
              m3 = fmaxf(m3, full || kk + 2 < lim ? sv[k + 2] : -INFINITY);
              m4 = fmaxf(m4, full || kk + 3 < lim ? sv[k + 3] : -INFINITY);
            }
          }
          m2 = fmaxf(fmaxf(m0, m1), fmaxf(m3, m4)) * a.scale_log2;
#pragma unroll
          for (int h = 0; h < 2 && !dead; ++h) {
            float sv[64];
            tmem_ld32(tS + h * 64, sv);
            tmem_ld32(tS + h * 64 + 32, sv + 32);
            tmem_ld_wait();
            if (bf16)
              l += full ? softmax_store_p<true, true>(sv, h, a.scale_log2, m2, lim, tS)
                        : softmax_store_p<true, false>(sv, h, a.scale_log2, m2, lim, tS);
            else
              l += full ? softmax_store_p<false, true>(sv, h, a.scale_log2, m2, lim, tS)
                        : softmax_store_p<false, false>(sv, h, a.scale_log2, m2, lim, tS);
          }
        }
        tmem_st_wait();            // P is in TMEM
        fence_proxy_async_smem();  // the zeroed V rows are visible to the MMA
        tc_fence_before();
        mbar_arrive(&c.p_full[grp]);
        pend = RowState{(size_t)et0 * a.G, m2, l, rows};
        pend_j = j;
      }
    }
    if (ok && pend_j >= 0) {
      ok = warp_all(
          mbar_wait(&c.o_full[grp], (pend_j >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
      if (ok) {
        tc_fence_after();
        ok = epilogue();
      }
    }
    // q rows requested by TMA have landed before the CTA may exit (after an
    // abort the issuer may not have waited for them)
    if (jq >= 0 && (warp & 3) == 0 && wl == 0)
      mbar_drain(&c.q_full[grp], (jq >> 1) & 1, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// The forward: each CTA runs its decode items (decode_body),
// then its KV-stationary items (all warps), in one launch.  TMEM (512
// columns) is allocated once for both phases.
template <int kKV>
__global__ void __launch_bounds__(kThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
          const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmqs, FwdArgs a,
          dec::DecArgs d) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint32_t s_tmem;
  const int warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  pdl_wait();  // the schedule (and the previous step's combine) are complete
  if (a.sch_hdr[kSchCtas] != (int)gridDim.x) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(a.flags, MXSA_FLAG_SCHEDULE);
    return;
  }
  const int b = blockIdx.x;
  const bool has_dec = d.cta_ptr != nullptr && d.cta_ptr[b] < d.cta_ptr[b + 1];
  const bool has_kvs = a.sch_hdr[kSchItems] > 0;  // claimed dynamically by every CTA
  if (!has_dec && !has_kvs) return;  // uniform: nothing to do, nothing allocated
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (has_dec) dec::decode_body<16, kKV>(tmk, tmv, tmq, d, sm, tmem);
  if (has_kvs) kv_stationary_body<kKV>(tmk, tmv, tmqs, a, sm, tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  if (has_kvs && threadIdx.x == 0) {
    // the last CTA to leave resets the claim counter for the next forward on
    // the same schedule (every CTA has finished claiming by now)
    __threadfence();
    if (atomicAdd(a.sch_hdr_mut + kSchExit, 1) == (int)gridDim.x - 1) {
      a.sch_hdr_mut[kSchClaim] = 0;
      a.sch_hdr_mut[kSchExit] = 0;
      __threadfence();
    }
  }
}

// 3-D view of a cache [pages * Hkv][page_size][128]: box = one page, one
// 128-byte column slab (64 x 16-bit, swizzled) or the full 128 e4m3 row.

bool make_cache_map(CUtensorMap* m, const void* base, const mxsa_problem& p) {
  auto fn = dec::encode_fn();
  if (!fn) return false;
  if (p.kv_dtype == MXSA_NVFP4) {
    // the code rows of the NVFP4 slabs [pages * Hkv][page_size * 72 bytes]:
    // box = one page's page_size rows of 64 bytes (the scale rows after
    // them come by bulk copy)
    cuuint64_t dims[3] = {64, (cuuint64_t)p.page_size, (cuuint64_t)p.num_pages * p.num_kv_heads};
    cuuint64_t strides[2] = {64, 72 * (cuuint64_t)p.page_size};
    cuuint32_t box[3] = {64u, (cuuint32_t)p.page_size, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  }
  const bool fp8 = p.kv_dtype == MXSA_FP8_E4M3;
  const cuuint64_t es = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {128, (cuuint64_t)p.page_size, (cuuint64_t)p.num_pages * p.num_kv_heads};
  cuuint64_t strides[2] = {128 * es, 128 * es * (cuuint64_t)p.page_size};
  cuuint32_t box[3] = {fp8 ? 128u : 64u, (cuuint32_t)p.page_size, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                               : (p.kv_dtype == MXSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// dynamic shared memory of the forward: the larger of its two phases' needs
size_t fwd_smem_bytes(bool fp8) {
  return std::max((size_t)(fp8 ? kCtrlFp8 : kCtrlBf16) + sizeof(Ctrl) + 1024, dec::smem_bytes(fp8));
}

cudaError_t launch_fwd(const mxsa_problem& p, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const IndexPtrs& ix, const SchedPtrs& sc, int num_ctas,
                       void* part_o, float* part_lse, cudaStream_t st, int* err_detail) {
  CUtensorMap tmk, tmv;
  if (!make_cache_map(&tmk, k_cache, p) || !make_cache_map(&tmv, v_cache, p)) {
    *err_detail = 1;
    return cudaErrorInvalidValue;
  }
  // one launch for both work lists (decode runs, KV-stationary tiles)
  dec::DecArgs d;
  CUtensorMap tmq;
  if (!dec::make_args(p, q, k_cache, v_cache, block_tables, ix, sc, part_o, part_lse, &d, &tmq)) {
    *err_detail = 1;
    return cudaErrorInvalidValue;
  }
  const bool fp8 = kv_widened(p);  // FP8 or NVFP4: staged and widened
  const size_t smem = fwd_smem_bytes(fp8);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    const int bytes = (int)std::max(fwd_smem_bytes(true), fwd_smem_bytes(false));
    attr_err = cudaFuncSetAttribute(k_fwd<dec::kKv16>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k_fwd<dec::kKvFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k_fwd<dec::kKvFp4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  FwdArgs a;
  a.q = static_cast<const uint8_t*>(q);
  a.block_tables = block_tables;
  a.seq = ix.seq;
  a.token_seq = ix.token_seq;
  a.entries = ix.entries;
  a.items = sc.items;
  a.cta_ptr = sc.cta_ptr;
  a.idx_hdr = ix.hdr;
  a.sch_hdr = sc.hdr;
  a.sch_hdr_mut = sc.hdr;
  a.claim = sc.hdr + kSchClaim;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.part32 = partials_fp32(p) ? 1 : 0;
  a.flags = ix.hdr + kHdrFlags;
  // q rows of the KV-stationary tiles: a box of one entry's G rows when G
  // is a multiple of 8 (whole swizzle atoms), else the warps' gather
  const int G = p.num_q_heads / p.num_kv_heads;
  CUtensorMap tmqs;
  std::memset(&tmqs, 0, sizeof(tmqs));
  a.q_tma = (G % 8 == 0 && G <= 128 && dec::make_q_map(&tmqs, q, p, G)) ? 1 : 0;
  a.num_seqs = p.num_seqs;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.topk = p.topk;
  a.page_size = p.page_size;
  a.max_pages = p.max_pages_per_seq;
  a.num_pages = p.num_pages;
  a.causal = p.causal;
  a.kv_fp8 = fp8 ? 1 : 0;
  a.kv_fp4 = p.kv_dtype == MXSA_NVFP4 ? 1 : 0;
  a.kbase = static_cast<const uint8_t*>(k_cache);
  a.vbase = static_cast<const uint8_t*>(v_cache);
  a.ab_bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
  a.per_tile = std::max(1, MXSA_TILE_ROWS / a.G);
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 0.08838834764831845f;  // 1/sqrt(128)
  a.scale_log2 = scale * 1.4426950408889634f;
  if (p.kv_dtype == MXSA_NVFP4)
    return launch_pdl(k_fwd<dec::kKvFp4>, dim3(num_ctas), dim3(kThreads), smem, st, tmk, tmv, tmq, tmqs, a, d);
  if (p.kv_dtype == MXSA_FP8_E4M3)
    return launch_pdl(k_fwd<dec::kKvFp8>, dim3(num_ctas), dim3(kThreads), smem, st, tmk, tmv, tmq, tmqs, a, d);
  return launch_pdl(k_fwd<dec::kKv16>, dim3(num_ctas), dim3(kThreads), smem, st, tmk, tmv, tmq, tmqs, a, d);
}

}  // namespace mxsa
