// Dense paged attention forward: every key up to the sequence length (and
// the query's position when causal) -- the all-blocks-selected case of the
// block-sparse method, computed without partials or a combine.  The MSA
// project page (sourcepulse "How It Works" and "Highlighted Details") lists a
// dense FlashAttention (FMHA) path next to the sparse one; the arithmetic is
// the method's definition with every block selected: softmax(q k^T * scale) v
// and lse = log sum exp, over keys p < L (and p <= pos(t) when causal,
// pos(t) = L - Tq + i).
//
// Persistent kernel, one CTA per SM, 352 threads.  A tile is 2T tokens
// (T = 128 / G) x the G query heads of one kv head of one sequence: two
// 128-row halves, one per softmax group, that share every K/V block.
//   warps 0-3, 4-7  softmax groups: row r of a half is thread r of its group
//              and TMEM lane r.  Per 128-key block: S = q k^T (TMEM), a lazily
//              raised running maximum (raised only when a score passes it by
//              2^8; O in TMEM is then rescaled), P = exp2(S - m) written back
//              to TMEM over S, l += sum P.  After the last block o = O / l
//              goes straight to the output and lse to its [Hq, Tq] slot.
//              While one group runs its softmax, the tensor pipe runs the
//              other group's products.
//   warp 8     producer: each half's q rows (one 3-D TMA box per 64-column
//              half: 64 columns x G heads x T tokens) and each block's K and
//              V pages (TMA through block_tables) into a 2-stage ring.
//   warps 9, 10  MMA issuers, one per group (tcgen05.mma, cta_group::1,
//              M = N = 128, K = 16, FP32 accumulate): q k^T into the group's
//              S once its previous p v is done, then P V into its O with P as
//              the TMEM operand.  Issuer 1 starts each tile only once group
//              0 has its first P, so the groups work out of step.
// TMEM: S and O of each group (512 columns).  The tiles are visited in a
// fixed order (round robin over the CTAs, latest tokens first), so every
// role walks the same sequence without sharing a queue.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mxsa {

namespace {

constexpr int kDThreads = 352;
constexpr int kDProducer = 8, kDMma = 9;  // warps 9, 10: the issuers of groups 0, 1
constexpr uint32_t kDTile = 32768;        // 128 rows x 128 x 16-bit
constexpr uint32_t kDStage = 2 * kDTile;  // K and V of one 128-token block
constexpr int kDMaxSeqs = 1024;           // sequences held in shared memory
constexpr float kDRescale = 8.f;          // log2 units

constexpr uint32_t kDOffQ = 0;            // 2 groups x q half
constexpr uint32_t kDOffKV = 2 * kDTile;
constexpr uint32_t kDOffSeq = kDOffKV + 2 * kDStage;

struct DCtrl {
  // q_*, s_full, p_*, o_*: one per softmax group; kv_*: per ring stage
  uint64_t q_full[2], q_empty[2], kv_full[2], kv_empty[2], s_full[2], p_full[2], p_empty[2], o_full[2], o_empty[2],
      done, go1;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t total_tiles, per_head;
  int32_t local_flags;  // the waits' status word when the caller passes none
};
constexpr uint32_t kDOffCtrl = kDOffSeq + kDMaxSeqs * 16;

struct DSeq {
  int32_t q_begin, tq, L, tiles_before;  // tiles_before: the tiles of earlier sequences (per kv head)
};

struct DenseArgs {
  const int32_t* block_tables;
  const int64_t* cu;
  const int32_t* lens;
  uint8_t* out;
  float* lse;
  int32_t* flags;  // may be null
  int32_t num_seqs, total_q, Hq, Hkv, G, T, page_size, max_pages, num_pages, causal, ab_bf16;
  float scale_log2;
};

__device__ __forceinline__ uint32_t dswz(uint32_t row, uint32_t chunk16) {
  return (chunk16 >> 3) * 16384u + row * 128u + (((chunk16 & 7u) ^ (row & 7u)) << 4);
}

template <bool kBf16>
__device__ __forceinline__ uint32_t dpack2(float a, float b) {
  if (kBf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// max of three floats in one instruction (NaN operands are ignored, as by fmaxf)
__device__ __forceinline__ float dmax3(float x, float y, float z) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
  return r;
}

__device__ __forceinline__ bool dwarp_all(bool v) { return __all_sync(0xffffffffu, v); }

// The tile the CTA visits n-th: tiles are numbered latest tokens first
// (their key ranges are the longest under causal masking), and CTA b takes
// numbers b, b + gridDim.x, ...  Returns false past the CTA's last tile.
struct DTile {
  int s, g, t0, ntok, nb;  // ntok: tokens of both halves (half h holds t0 + hT ..)
};

__device__ __forceinline__ bool dense_tile(const DSeq* seq, const DCtrl& c, const DenseArgs& a, int n, DTile* d) {
  const long long idx = (long long)blockIdx.x + (long long)n * gridDim.x;
  if (idx >= c.total_tiles) return false;
  const int i = c.total_tiles - 1 - (int)idx;
  const int g = i / c.per_head, rem = i - g * c.per_head;
  int lo = 0, hi = a.num_seqs - 1;  // last sequence with tiles_before <= rem
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seq[mid].tiles_before <= rem) lo = mid;
    else hi = mid - 1;
  }
  const DSeq sq = seq[lo];
  d->s = lo;
  d->g = g;
  d->t0 = (rem - sq.tiles_before) * 2 * a.T;
  d->ntok = min(2 * a.T, sq.tq - d->t0);
  const int nblk = (sq.L + 127) >> 7;
  if (a.causal) {
    const int last = sq.L - sq.tq + d->t0 + d->ntok - 1;  // position of the tile's last token
    d->nb = last < 0 ? 0 : min(nblk, (last >> 7) + 1);
  } else {
    d->nb = nblk;
  }
  return true;
}

// P = exp2(S * scale_log2 - m) of one row over keys 64h .. 64h + 63 (masked
// to k < lim unless kFull: every key visible), packed in pairs and written
// to TMEM columns tP + 32h ..; returns the partial row sum.
template <bool kFull, bool kBf16>
__device__ __forceinline__ float dense_p(const float* sv, int h, float scale_log2, float m, int lim, uint32_t tP) {
  float l0 = 0.f, l1 = 0.f;
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int k0 = 64 * h + 2 * i;
    float p0 = ex2_approx(fmaf(sv[2 * i], scale_log2, -m));
    float p1 = ex2_approx(fmaf(sv[2 * i + 1], scale_log2, -m));
    if (!kFull) {
      p0 = k0 < lim ? p0 : 0.f;
      p1 = k0 + 1 < lim ? p1 : 0.f;
    }
    if (i & 1) l1 += p0 + p1;
    else l0 += p0 + p1;
    pk[i] = dpack2<kBf16>(p0, p1);
  }
  tmem_st32(tP + 32 * h, pk);
  return l0 + l1;
}

template <bool kBf16>
__global__ void __launch_bounds__(kDThreads, 1)
    k_dense(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
            const __grid_constant__ CUtensorMap tmv, DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DSeq* seq = reinterpret_cast<DSeq*>(sm + kDOffSeq);
  DCtrl& c = *reinterpret_cast<DCtrl*>(sm + kDOffCtrl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  pdl_wait();

  // sequence table: q_begin, tq, L (clamped) and the tiles before each
  // sequence; a sequence whose cu_seqlens_q entries are out of order or past
  // total_q gets no tokens
  const int B = a.num_seqs;
  const int maxL = a.max_pages * a.page_size;
  for (int s = tid; s < B; s += kDThreads) {
    const long long b0 = a.cu[s], b1 = a.cu[s + 1];
    const bool ok = b0 >= 0 && b1 >= b0 && b1 <= a.total_q;
    DSeq d;
    d.q_begin = ok ? (int)b0 : 0;
    d.tq = ok ? (int)(b1 - b0) : 0;
    d.L = min(max(a.lens[s], 0), maxL);
    d.tiles_before = (d.tq + 2 * a.T - 1) / (2 * a.T);  // this sequence's own tiles for now
    seq[s] = d;
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;  // exclusive prefix (B <= 1024: one serial pass)
    for (int s = 0; s < B; ++s) {
      const int n = seq[s].tiles_before;
      seq[s].tiles_before = run;
      run += n;
    }
    c.per_head = run;
    c.total_tiles = run * a.Hkv;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c.q_full[i], 1);
      mbar_init(&c.q_empty[i], 1);
      mbar_init(&c.kv_full[i], 1);
      mbar_init(&c.kv_empty[i], 2);  // both issuers' p v of the block
      mbar_init(&c.s_full[i], 1);
      mbar_init(&c.p_full[i], 128);
      mbar_init(&c.p_empty[i], 1);
      mbar_init(&c.o_full[i], 1);
      mbar_init(&c.o_empty[i], 128);
    }
    mbar_init(&c.done, 2);
    mbar_init(&c.go1, 1);
    c.abort_flag = 0;
    c.local_flags = 0;
    fence_mbar_init();
  }
  if (warp == kDMma) {
    tmem_alloc(&c.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  volatile int* abort_flag = &c.abort_flag;
  int32_t* const fl = a.flags ? a.flags : &c.local_flags;
  const uint32_t sbase = smem_u32(sm);
  const int G = a.G;

  if (blockIdx.x < c.total_tiles) {
    if (warp == kDProducer) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        const int ps = a.page_size, npg = ps == 128 ? 1 : 2;
        int blk = 0, n = 0;
        bool ok = true;
        DTile d;
        for (; ok && dense_tile(seq, c, a, n, &d); ++n) {
          const DSeq sq = seq[d.s];
          for (int h = 0; h < 2 && ok; ++h) {
            // half h's rows (its tokens may run past the sequence: those rows
            // are padding, never stored)
            ok = mbar_wait(&c.q_empty[h], (n & 1) ^ 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (!ok) break;
            uint8_t* qd = sm + kDOffQ + h * kDTile;
            mbar_arrive_expect_tx(&c.q_full[h], (uint32_t)(G * a.T) * 256u);
            tma_load_3d(qd, &tmq, &c.q_full[h], 0, d.g * G, sq.q_begin + d.t0 + h * a.T);
            tma_load_3d(qd + 16384, &tmq, &c.q_full[h], 64, d.g * G, sq.q_begin + d.t0 + h * a.T);
          }
          if (!ok) break;
          for (int b = 0; b < d.nb && ok; ++b, ++blk) {
            const int st = blk & 1, us = blk >> 1;
            ok = mbar_wait(&c.kv_empty[st], (us & 1) ^ 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (!ok) break;
            const int valid = min(128, sq.L - 128 * b);
            int pages[2] = {-1, -1};
            for (int pg = 0; pg < npg; ++pg) {
              if (pg * 64 >= valid) continue;
              const int lp = ps == 128 ? b : 2 * b + pg;
              const int phys = a.block_tables[(size_t)d.s * a.max_pages + lp];
              if (phys < 0 || phys >= a.num_pages) {
                atomicOr(fl, MXSA_FLAG_PAGE);
                continue;
              }
              pages[pg] = phys;
            }
            const int present = (pages[0] >= 0) + (pages[1] >= 0);
            uint8_t* kdst = sm + kDOffKV + st * kDStage;
            uint8_t* vdst = kdst + kDTile;
            mbar_arrive_expect_tx(&c.kv_full[st], (uint32_t)present * (uint32_t)ps * 512u);
            for (int pg = 0; pg < npg; ++pg) {
              if (pages[pg] < 0) continue;
              const int z = pages[pg] * a.Hkv + d.g;
              for (int h = 0; h < 2; ++h) {
                tma_load_3d(kdst + h * 16384 + pg * 8192, &tmk, &c.kv_full[st], h * 64, 0, z);
                tma_load_3d(vdst + h * 16384 + pg * 8192, &tmv, &c.kv_full[st], h * 64, 0, z);
              }
            }
          }
        }
        // drain: the copies in flight land before the CTA may exit
        for (int k = std::max(0, blk - 2); k < blk; ++k)
          mbar_drain(&c.kv_full[k & 1], (k >> 1) & 1, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        if (n > 0)
          for (int h = 0; h < 2; ++h) mbar_drain(&c.q_full[h], (n - 1) & 1, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
      }
    } else if (warp == kDMma || warp == kDMma + 1) {
      // --------------------------------------------------------- MMA issuers
      // Issuer g serves softmax group g: its S is overwritten only once its
      // previous p v (which read P from it) is done, so by the time the group
      // sees S its O is complete too.
      if (lane == 0) {
        const int gq = warp - kDMma;
        const uint32_t id_qk = idesc_f16(128, 128, kBf16 ? 1u : 0u, 0, 0);
        const uint32_t id_pv = idesc_f16(128, 128, kBf16 ? 1u : 0u, 0, 1);
        const uint32_t q_s = sbase + kDOffQ + gq * kDTile;
        const uint32_t tS = tmem + gq * 256, tO = tS + 128;
        int blk = 0, n = 0, ng = 0;
        bool ok = true;
        DTile d;
        for (; ok && dense_tile(seq, c, a, n, &d); ++n) {
          ok = mbar_wait(&c.q_full[gq], n & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (!ok) break;
          if (d.nb == 0) mma_commit(&c.q_empty[gq]);  // q unused: free at once
          if (d.nb == 0 && n > 0) {
            // no p v of this tile waits for the previous tile's epilogue, so
            // wait here: o_full must not complete twice before the group has
            // read the first completion (its parity wait would miss it)
            ok = mbar_wait(&c.o_empty[gq], (n - 1) & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (!ok) break;
          }
          if (gq == 1 && d.nb > 0) {
            // group 1 starts a tile once group 0 has its first P, so the two
            // groups' softmax and MMAs alternate instead of running in step
            // (go1 completes once per tile with blocks; issuer 0 cannot run a
            // tile ahead: its next tile needs this issuer's last p v)
            ok = mbar_wait(&c.go1, ng & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            ++ng;
            if (!ok) break;
          }
          for (int b = 0; b < d.nb && ok; ++b, ++blk) {
            const int st = blk & 1;
            ok = mbar_wait(&c.kv_full[st], (blk >> 1) & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (!ok) break;
            if (blk > 0) {  // the previous p v read P from S
              ok = mbar_wait(&c.p_empty[gq], (blk - 1) & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
              if (!ok) break;
            }
            tc_fence_after();
            const uint32_t k_s = sbase + kDOffKV + st * kDStage, v_s = k_s + kDTile;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
              mma_f16_ss(tS, smem_desc_sw128(q_s + off, 0, 1024), smem_desc_sw128(k_s + off, 0, 1024), id_qk,
                         ks > 0);
            }
            if (b == d.nb - 1) mma_commit(&c.q_empty[gq]);  // the half's q is read once these complete
            mma_commit(&c.s_full[gq]);
            ok = mbar_wait(&c.p_full[gq], blk & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (!ok) break;
            if (gq == 0 && b == 0) mbar_arrive(&c.go1);
            if (b == 0 && n > 0) {  // O of the previous tile has been read out
              ok = mbar_wait(&c.o_empty[gq], (n - 1) & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
              if (!ok) break;
            }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_f16_ts(tO, tS + ks * 8, smem_desc_sw128(v_s + ks * 2048u, 16384, 1024), id_pv,
                         (b > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&c.p_empty[gq]);
            mma_commit(&c.kv_empty[st]);
          }
          if (ok) mma_commit(&c.o_full[gq]);
        }
        mma_commit(&c.done);
        mbar_drain(&c.done, 0, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
      }
    } else {
      // ------------------------------------------------------------- softmax
      const int gq = warp >> 2;  // softmax group: the tile's half
      const int r = tid & 127;   // row of the half == TMEM lane
      const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tO = tmem + gq * 256 + 128 + lane_addr;
      const int tt = gq * a.T + r / G, hh = r % G;  // token within the tile, head within the group
      int blk = 0, n = 0;
      bool ok = true;
      DTile d;
      for (; ok && dense_tile(seq, c, a, n, &d); ++n) {
        const DSeq sq = seq[d.s];
        const bool live = r < G * a.T && tt < d.ntok;  // rows past G*T are padding of the half
        const int pos = sq.L - sq.tq + d.t0 + tt;
        float m = -INFINITY, l = 0.f;
        for (int b = 0; b < d.nb && ok; ++b, ++blk) {
          const int st = blk & 1;
          ok = dwarp_all(mbar_wait(&c.s_full[gq], blk & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
          const int valid = min(128, sq.L - 128 * b);
          int lim = live ? valid : 0;
          if (a.causal) lim = min(lim, pos - 128 * b + 1);
          const uint32_t tS = tmem + gq * 256 + lane_addr;
          // block maximum (log2 units); a warp whose rows all see every key
          // of the block skips the masking
          const bool full = __all_sync(0xffffffffu, lim >= 128);
          float b0 = -INFINITY, b1 = -INFINITY, b2 = -INFINITY, b3 = -INFINITY;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float sv[64];
            tmem_ld32(tS + h * 64, sv);
            tmem_ld32(tS + h * 64 + 32, sv + 32);
            tmem_ld_wait();
            if (full) {
#pragma unroll
              for (int k = 0; k < 64; k += 8) {
                b0 = dmax3(b0, sv[k], sv[k + 1]);
                b1 = dmax3(b1, sv[k + 2], sv[k + 3]);
                b2 = dmax3(b2, sv[k + 4], sv[k + 5]);
                b3 = dmax3(b3, sv[k + 6], sv[k + 7]);
              }
            } else {
#pragma unroll
              for (int k = 0; k < 64; k += 4) {
                const int kk = 64 * h + k;
                b0 = fmaxf(b0, kk < lim ? sv[k] : -INFINITY);
                b1 = fmaxf(b1, kk + 1 < lim ? sv[k + 1] : -INFINITY);
                b2 = fmaxf(b2, kk + 2 < lim ? sv[k + 2] : -INFINITY);
                b3 = fmaxf(b3, kk + 3 < lim ? sv[k + 3] : -INFINITY);
              }
            }
          }
          const float bm = fmaxf(fmaxf(b0, b1), fmaxf(b2, b3)) * a.scale_log2;
          const bool raise = bm > m + kDRescale || (m == -INFINITY && bm > -INFINITY);
          if (__any_sync(0xffffffffu, raise)) {
            const float f = raise ? (m == -INFINITY ? 0.f : ex2_approx(m - bm)) : 1.f;
            if (b > 0) {
              // O holds this tile's blocks so far and is complete: the
              // issuer overwrote S only after the last p v into O was done
#pragma unroll
              for (int cb = 0; cb < 4; ++cb) {
                float ov[32];
                tmem_ld32(tO + cb * 32, ov);
                tmem_ld_wait();
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(ov[i] * f);
                tmem_st32(tO + cb * 32, w);
              }
            }
            if (raise) {
              l *= f;
              m = bm;
            }
          }
          // P over the S columns, l
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float sv[64];
            tmem_ld32(tS + h * 64, sv);
            tmem_ld32(tS + h * 64 + 32, sv + 32);
            tmem_ld_wait();
            const float mm = m == -INFINITY ? 0.f : m;
            l += full ? dense_p<true, kBf16>(sv, h, a.scale_log2, mm, lim, tS)
                      : dense_p<false, kBf16>(sv, h, a.scale_log2, mm, lim, tS);
          }
          if (valid < 128 && r >= valid) {
            // keys past the sequence end: zero V rows (stale values may be
            // NaN bit patterns, and 0 * NaN would reach O); the writer's
            // proxy fence orders them before the p v that reads them
            const uint32_t vs = sbase + kDOffKV + st * kDStage + kDTile;
            for (int ch = 0; ch < 16; ++ch) st_shared_v4(vs + dswz(r, ch), 0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&c.p_full[gq]);
        }
        if (!ok) break;
        // ---- the tile's output rows
        ok = dwarp_all(mbar_wait(&c.o_full[gq], n & 1, abort_flag, fl, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        uint8_t* orow = a.out + ((size_t)(sq.q_begin + d.t0 + tt) * a.Hq + (size_t)d.g * G + hh) * 256;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          float ov[32];
          tmem_ld32(tO + cb * 32, ov);  // every lane: the load is warp-collective
          tmem_ld_wait();
          if (live) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = d.nb > 0 ? dpack2<kBf16>(ov[2 * i] * inv_l, ov[2 * i + 1] * inv_l) : 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(orow + cb * 64 + i * 16) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2],
                                                                              w[4 * i + 3]);
          }
        }
        if (live && a.lse)
          a.lse[(size_t)(d.g * G + hh) * a.total_q + sq.q_begin + d.t0 + tt] =
              l > 0.f ? (m + lg2_approx(l)) * 0.69314718055994530942f : -INFINITY;
        tc_fence_before();
        mbar_arrive(&c.o_empty[gq]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kDMma) tmem_dealloc(tmem, 512);
}

bool dense_kv_map(CUtensorMap* m, const void* base, const mxsa_problem& p, PFN_cuTensorMapEncodeTiled_v12000 fn) {
  cuuint64_t dims[3] = {128, (cuuint64_t)p.page_size, (cuuint64_t)p.num_pages * p.num_kv_heads};
  cuuint64_t strides[2] = {256, 256 * (cuuint64_t)p.page_size};
  cuuint32_t box[3] = {64, (cuuint32_t)p.page_size, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      p.kv_dtype == MXSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 dense_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

size_t dense_smem_bytes() { return kDOffCtrl + sizeof(DCtrl) + 1024; }

}  // namespace

cudaError_t launch_dense(const mxsa_problem& p, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int64_t* cu, const int32_t* lens, void* out, float* lse,
                         int32_t* flags, cudaStream_t st) {
  if (p.total_q == 0) return cudaSuccess;
  auto fn = dense_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const int G = p.num_q_heads / p.num_kv_heads, T = 128 / G;
  CUtensorMap tmq, tmk, tmv;
  // q viewed as [total_q][Hq][128]: one box = 64 columns x G heads x T tokens
  cuuint64_t qd[3] = {128, (cuuint64_t)p.num_q_heads, (cuuint64_t)p.total_q};
  cuuint64_t qs[2] = {256, 256 * (cuuint64_t)p.num_q_heads};
  cuuint32_t qb[3] = {64, (cuuint32_t)G, (cuuint32_t)T};
  cuuint32_t qe[3] = {1, 1, 1};
  const CUtensorMapDataType qt =
      p.q_dtype == MXSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (fn(&tmq, qt, 3, const_cast<void*>(q), qd, qs, qb, qe, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS ||
      !dense_kv_map(&tmk, k_cache, p, fn) || !dense_kv_map(&tmv, v_cache, p, fn))
    return cudaErrorInvalidValue;
  DenseArgs a;
  a.block_tables = block_tables;
  a.cu = cu;
  a.lens = lens;
  a.out = static_cast<uint8_t*>(out);
  a.lse = lse;
  a.flags = flags;
  a.num_seqs = p.num_seqs;
  a.total_q = p.total_q;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = G;
  a.T = T;
  a.page_size = p.page_size;
  a.max_pages = p.max_pages_per_seq;
  a.num_pages = p.num_pages;
  a.causal = p.causal;
  a.ab_bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
  auto* kern = a.ab_bf16 ? k_dense<true> : k_dense<false>;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 0.08838834764831845f;  // 1/sqrt(128)
  a.scale_log2 = scale * 1.4426950408889634f;
  const size_t smem = dense_smem_bytes();
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [smem] {
    attr_err = cudaFuncSetAttribute(k_dense<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k_dense<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(kern, dim3(sms), dim3(kDThreads), smem, st, tmq, tmk, tmv, a);
}

}  // namespace mxsa
