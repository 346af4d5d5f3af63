// Top-k block selection: the step before the index, which 128-token blocks
// each (token, kv head) row attends to.  The MSA summary page ("How It
// Works") names the "sparse top-k selection"; the sglang pull request
// ("Summary") writes an index K cache beside K and V.  The pages give no
// scoring rule; the library's reading:
//   dot(t, g, p)   = FP32 sum of iq[t][g][d] * ik[p][g][d], fused multiply-
//                    adds in the order d = 0 .. D-1 from +0 (NaN: skipped);
//   score(t, g, b) = max of dot over the block's visible positions (p < L,
//                    p <= pos(t) when causal, p on a valid page);
//   sel[t][g][:]   = the blocks with a score by (score descending, block
//                    ascending), the first topk; the rest -1.
// The selection is an integer decision, so the kernels compute exactly that
// arithmetic (CUDA-core FMAs in dimension order, exact maxima and an exact
// sort); the result is bit-identical to a plain CPU statement of it.
//
// Four launches, chained by programmatic dependent launch:
//   k_select_prep   one CTA: per sequence its clamped length, first token,
//                   new tokens and blocks, and the exclusive prefixes of
//                   the two kinds of work units (below), into the workspace.
//   k_select_short  units (sequence, block, kv head) of the sequences with at
//                   most 8 new tokens: the block's key rows are staged in
//                   shared memory by coalesced 16-byte loads, thread p walks
//                   row p and the block's maximum per query comes from a CTA
//                   reduction.  The index keys are read once: this is the
//                   HBM-bound decode case, so the kernel keeps few registers
//                   and little shared memory, for many CTAs per SM.
//   k_select_long   units (sequence, block, kv head, 128-query chunk) of the
//                   longer sequences: the chunk's queries and the block's keys
//                   staged as FP32, 32 dimensions at a time, and multiplied
//                   like a matrix product (8 x 8 accumulators per thread),
//                   then a maximum over each query's visible keys.
//   k_select_topk   one CTA per (token, kv head) row: the row's block scores
//                   become 64-bit keys (order-preserving score bits above the
//                   complemented block index) in shared memory, sorted by a
//                   bitonic network, and the first topk blocks are written.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace mxsa {

namespace {

constexpr int kSelThreads = 128;
constexpr int kPrepThreads = 1024;   // one sequence per thread
constexpr int kSelMaxBlocks = 4096;  // blocks per sequence (the sort buffer)
constexpr int kSelSmallTq = 8;       // at most this many new tokens: the short form
constexpr int kTopkThreads = 256;

// The sequence table k_select_prep writes after the scores.
struct SeqRec {
  int32_t L, q0, tq, nblk;
};

struct SelTable {
  SeqRec* seq;             // [B]
  long long* unit_short;   // [B + 1] exclusive prefix of short units
  long long* unit_long;    // [B + 1] exclusive prefix of long units
  int32_t* bad;            // cu_seqlens_q is not a non-decreasing partition
};

struct SelArgs {
  const uint8_t* iq;        // [total_q][Hkv][D]
  const uint8_t* ik;        // [pages][Hkv][ps][D]
  const int32_t* bt;
  const int64_t* cu;
  const int32_t* lens;
  float* score;             // [total_q][Hkv][max_blocks]
  int32_t* sel;             // [total_q][Hkv][topk]
  int32_t* flags;           // may be null
  SelTable tab;
  int32_t B, total_q, Hkv, D, ps, num_pages, max_pages, max_blocks, topk, causal, dtype;
};

// The values of one 16-byte chunk, widened exactly to FP32 in dimension
// order: 16 e4m3 values, or 8 of a 16-bit type.
__device__ __forceinline__ void unpack_e4m3x16(uint4 v, float* out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(w[i] >> (16 * h))));
      const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h2));
      out[4 * i + 2 * h] = f.x;
      out[4 * i + 2 * h + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void unpack_16bitx8(uint4 v, bool bf16, float* out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (bf16) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
}

// last s in [0, B) with prefix[s] <= v (prefix non-decreasing, prefix[0] = 0;
// a sequence without units shares its start with the next one, which wins)
__device__ __forceinline__ int unit_seq(const long long* prefix, int B, long long v) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPrepThreads) k_select_prep(SelArgs a) {
  __shared__ long long s_part[2][kPrepThreads / 32];
  __shared__ int s_bad;
  pdl_launch_dependents();
  pdl_wait();  // the previous user of the workspace is done
  const int s = threadIdx.x, lane = s & 31, warp = s >> 5;
  if (s == 0) s_bad = (a.cu[0] != 0 || a.cu[a.B] != a.total_q) ? 1 : 0;
  __syncthreads();
  long long nshort = 0, nlong = 0;
  if (s < a.B) {
    const long long cap = (long long)a.max_pages * a.ps;
    const long long c0 = a.cu[s], c1 = a.cu[s + 1];
    if (c1 < c0) s_bad = 1;
    long long L = a.lens[s];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int tq = (int)(c1 > c0 ? c1 - c0 : 0);
    const int nb = (int)((L + 127) / 128);
    a.tab.seq[s] = SeqRec{(int)L, (int)c0, tq, nb};
    if (tq >= 1 && tq <= kSelSmallTq) nshort = nb;
    if (tq > kSelSmallTq) nlong = (long long)nb * ((tq + kSelThreads - 1) / kSelThreads);
  }
  // block-wide exclusive scans of both unit counts
  long long is = nshort, il = nlong;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long xs = __shfl_up_sync(0xffffffffu, is, o), xl = __shfl_up_sync(0xffffffffu, il, o);
    if (lane >= o) {
      is += xs;
      il += xl;
    }
  }
  if (lane == 31) {
    s_part[0][warp] = is;
    s_part[1][warp] = il;
  }
  __syncthreads();
  if (s == 0) {
    long long as = 0, al = 0;
    for (int w = 0; w < kPrepThreads / 32; ++w) {
      const long long vs = s_part[0][w], vl = s_part[1][w];
      s_part[0][w] = as;
      s_part[1][w] = al;
      as += vs;
      al += vl;
    }
    a.tab.unit_short[a.B] = as;
    a.tab.unit_long[a.B] = al;
  }
  __syncthreads();
  if (s < a.B) {
    a.tab.unit_short[s] = s_part[0][warp] + is - nshort;
    a.tab.unit_long[s] = s_part[1][warp] + il - nlong;
  }
  if (s == 0) {
    *a.tab.bad = s_bad;
    if (s_bad) {  // nothing is scored: every row will be -1
      a.tab.unit_short[a.B] = 0;
      a.tab.unit_long[a.B] = 0;
      if (a.flags) atomicOr(a.flags, MXSA_FLAG_CU);
    }
  }
}

// k_select_short: each unit's key rows come into a ring of kShortStages
// shared-memory stages by TMA tiled copies (one box per page slice and
// 128-byte column segment, swizzled: 16-byte chunk c of row r of a
// segment lands at chunk c ^ (r & 7) for 128-byte rows, c ^ ((r >> 1) & 3)
// for 64-byte ones), and the unit's query rows by bulk copies.  Thread 0
// issues them kShortStages - 1 units ahead, so later units' copies overlap
// this unit's scoring.  Thread r reads row r chunk by chunk in dimension
// order; the swizzle spreads any 8 consecutive rows' same chunk over all
// banks.
constexpr int kShortStages = 3;

// bytes of one row segment in shared memory (the swizzle span) and stage size
__host__ __device__ constexpr int short_span(int D, int esz) { return D * esz < 128 ? D * esz : 128; }
__host__ __device__ constexpr size_t short_stage_bytes(int D, int esz) {
  return ((size_t)(kSelThreads + kSelSmallTq) * D * esz + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr size_t short_smem(int D, int esz) {
  return kShortStages * short_stage_bytes(D, esz) + 1024;  // + alignment of the base to 1024
}

// What a short unit is: its sequence record, block and kv head.
struct ShortUnit {
  SeqRec r;
  int s, b, g;
};

// A staged unit as the producer warp describes it to the scoring warps.
struct ShortInfo {
  int b, g, tq, L, q0, pg_lo, pg_hi;  // pages of key rows 0-63 and 64-127 (-1: none)
  int pad;
};

// Page of the unit block's key row rr (0..127), or -1 (past the sequence or
// outside [0, num_pages)).
__device__ __forceinline__ int short_page(const SelArgs& a, const ShortUnit& x, int rr) {
  const int key = 128 * x.b + rr;
  if (key >= x.r.L) return -1;
  const int pg = a.bt[(long long)x.s * a.max_pages + key / a.ps];
  return (pg >= 0 && pg < a.num_pages) ? pg : -1;
}

// The producer's look-ups for unit u: the sequence (advanced from *s_cur,
// the previous unit's: a CTA's units come in increasing order), the
// block's pages and the bytes its copies will bring.
struct ShortPlan {
  ShortInfo in;
  int s;
  uint32_t bytes;
};

__device__ __forceinline__ ShortPlan short_plan(const SelArgs& a, long long u, int* s_cur, int D, int esz) {
  ShortPlan pl;
  const int g = (int)(u % a.Hkv);
  const long long v = u / a.Hkv;
  int s = *s_cur;
  while (s + 1 < a.B && a.tab.unit_short[s + 1] <= v) ++s;  // the last s with prefix[s] <= v
  *s_cur = s;
  const SeqRec r = a.tab.seq[s];
  ShortUnit x;
  x.r = r;
  x.s = s;
  x.g = g;
  x.b = (int)(v - a.tab.unit_short[s]);
  const uint32_t row = (uint32_t)D * esz, span = (uint32_t)short_span(D, esz), nseg = row / span;
  const int n_slices = a.ps == 128 ? 1 : 2, per = a.ps == 128 ? 128 : 64;
  int pgs[2] = {-1, -1};
  uint32_t bytes = (uint32_t)r.tq * row;
  for (int h = 0; h < n_slices; ++h) {
    pgs[h] = short_page(a, x, per * h);
    if (pgs[h] >= 0) bytes += nseg * (uint32_t)per * span;
  }
  pl.in.b = x.b;
  pl.in.g = g;
  pl.in.tq = r.tq;
  pl.in.L = r.L;
  pl.in.q0 = r.q0;
  pl.in.pg_lo = pgs[0];
  pl.in.pg_hi = a.ps == 128 ? pgs[0] : pgs[1];
  pl.in.pad = 0;
  pl.s = s;
  pl.bytes = bytes;
  return pl;
}

// The copies of a planned unit into stage `st` on barrier `full`: per page
// slice of the block (one for 128-token pages, two for 64) on a valid page,
// one TMA box per column segment (segment sg of rows at sg * 128 * span +
// row * span); then the query rows after the 128 key rows.
__device__ __forceinline__ void short_issue(const SelArgs& a, const CUtensorMap* tmk, const ShortPlan& pl,
                                            uint8_t* st, uint64_t* full, ShortInfo* info, int D, int esz) {
  const uint32_t row = (uint32_t)D * esz, span = (uint32_t)short_span(D, esz), nseg = row / span;
  const int n_slices = a.ps == 128 ? 1 : 2, per = a.ps == 128 ? 128 : 64;
  *info = pl.in;  // published by the arrival below
  mbar_arrive_expect_tx(full, pl.bytes);
  for (int h = 0; h < n_slices; ++h) {
    const int pg = h == 0 ? pl.in.pg_lo : pl.in.pg_hi;
    if (pg < 0) continue;
    for (uint32_t sg = 0; sg < nseg; ++sg)
      tma_load_3d(st + (size_t)sg * kSelThreads * span + (size_t)per * h * span, tmk, full,
                  (int)(sg * span / esz), 0, pg * a.Hkv + pl.in.g);
  }
  for (int i = 0; i < pl.in.tq; ++i)
    bulk_load(st + (size_t)kSelThreads * row + (size_t)i * row,
              a.iq + ((long long)(pl.in.q0 + i) * a.Hkv + pl.in.g) * row, row, full);
}

// Dot products of key row t (swizzled segments in `keys`) with the first
// tq (<= NQ) query rows (plain rows in `qrows`), each summed by fused
// multiply-adds in dimension order.
template <int D, bool kFp8, int NQ>
__device__ __forceinline__ void short_dots(const uint8_t* keys, const uint8_t* qrows, int t, int tq, bool bf16,
                                           float* acc) {
  constexpr int esz = kFp8 ? 1 : 2, span = short_span(D, esz), nseg = D * esz / span, cps = span / 16;
  constexpr int epc = 16 / esz;  // elements per 16-byte chunk
#pragma unroll
  for (int sg = 0; sg < nseg; ++sg) {
#pragma unroll
    for (int c = 0; c < cps; ++c) {
      const int sw = span == 128 ? (c ^ (t & 7)) : (c ^ ((t >> 1) & 3));
      const uint4 kv = *reinterpret_cast<const uint4*>(keys + (size_t)sg * kSelThreads * span + (size_t)t * span + sw * 16);
      float kd[16];
      if (kFp8) unpack_e4m3x16(kv, kd);
      else unpack_16bitx8(kv, bf16, kd);
      const int dchunk = sg * cps + c;  // the chunk's place in the row
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        if (i >= tq) break;
        const uint4 qv = *reinterpret_cast<const uint4*>(qrows + (size_t)i * D * esz + dchunk * 16);
        float qd[16];
        if (kFp8) unpack_e4m3x16(qv, qd);
        else unpack_16bitx8(qv, bf16, qd);
#pragma unroll
        for (int e = 0; e < epc; ++e) acc[i] = __fmaf_rn(qd[e], kd[e], acc[i]);
      }
    }
  }
}

// 160 threads: warps 0-3 score (thread r: key row r), warp 4 issues the
// copies kShortStages units ahead.
constexpr int kShortThreads = kSelThreads + 32;

template <int D, bool kFp8>
__global__ void __launch_bounds__(kShortThreads)
    k_select_short(const __grid_constant__ CUtensorMap tmk, SelArgs a) {
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kShortStages], empty[kShortStages];
  __shared__ ShortInfo info[kShortStages];
  __shared__ float red_max[kSelSmallTq][kSelThreads / 32];
  __shared__ int red_have[kSelSmallTq][kSelThreads / 32];
  __shared__ int abort_flag, sink;
  pdl_wait();  // the sequence table
  // only now: k_select_long reads the table without a wait of its own
  pdl_launch_dependents();
  constexpr int esz = kFp8 ? 1 : 2;
  constexpr size_t stage = short_stage_bytes(D, esz);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bf16 = a.dtype == MXSA_BF16;
  const long long units = a.tab.unit_short[a.B] * a.Hkv;
  const long long first = blockIdx.x, stride = gridDim.x;
  if (first >= units) return;  // uniform
  const long long n_mine = (units - first + stride - 1) / stride;
  if (tid == 0) {
    for (int i = 0; i < kShortStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kSelThreads);
    }
    abort_flag = 0;
    sink = 0;
    fence_mbar_init();
  }
  __syncthreads();
  int* status = a.flags ? a.flags : &sink;
  if (warp == kSelThreads / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      int s_cur = 0;
      for (long long j = 0; j < n_mine; ++j) {
        const int st = (int)(j % kShortStages);
        // the look-ups first: their latency overlaps the wait for the stage
        const ShortPlan pl = short_plan(a, first + j * stride, &s_cur, D, esz);
        // the stage's previous unit (j - kShortStages) was scored
        if (!mbar_wait(&empty[st], (uint32_t)(((j / kShortStages) & 1) ^ 1), &abort_flag, status, MXSA_FLAG_TIMEOUT,
                       kWaitLimitNs))
          break;
        short_issue(a, &tmk, pl, sm + st * stage, &full[st], &info[st], D, esz);
      }
      // copies of the last units may still be in flight if a wait gave up
      for (long long i = n_mine > kShortStages ? n_mine - kShortStages : 0; i < n_mine; ++i)
        mbar_drain(&full[i % kShortStages], (uint32_t)((i / kShortStages) & 1), status, MXSA_FLAG_TIMEOUT,
                   kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------- scoring
    for (long long i = 0; i < n_mine; ++i) {
      const int st = (int)(i % kShortStages);
      const bool ok = mbar_wait(&full[st], (uint32_t)((i / kShortStages) & 1), &abort_flag, status,
                                MXSA_FLAG_TIMEOUT, kWaitLimitNs);
      const ShortInfo x = info[st];
      const int tq = ok ? x.tq : 0, L = x.L, q0 = x.q0, b = x.b;
      const int page = 128 * b + tid < L ? (tid < 64 ? x.pg_lo : x.pg_hi) : -1;
      float best[kSelSmallTq];
      int have[kSelSmallTq];
#pragma unroll
      for (int q = 0; q < kSelSmallTq; ++q) {
        best[q] = -INFINITY;
        have[q] = 0;
      }
      if (ok && page >= 0) {
        float acc[kSelSmallTq];
#pragma unroll
        for (int q = 0; q < kSelSmallTq; ++q) acc[q] = 0.f;
        const uint8_t* keys = sm + st * stage;
        const uint8_t* qrows = keys + (size_t)kSelThreads * D * esz;
        if (tq == 1) short_dots<D, kFp8, 1>(keys, qrows, tid, 1, bf16, acc);
        else short_dots<D, kFp8, kSelSmallTq>(keys, qrows, tid, tq, bf16, acc);
        const int p = 128 * b + tid;
#pragma unroll
        for (int q = 0; q < kSelSmallTq; ++q) {
          const int pos = L - tq + q;
          if (q < tq && (!a.causal || p <= pos) && !isnan(acc[q])) {
            best[q] = acc[q];
            have[q] = 1;
          }
        }
      }
      mbar_arrive(&empty[st]);  // this thread is done with the stage
#pragma unroll
      for (int q = 0; q < kSelSmallTq; ++q) {
        if (q >= tq) break;
        float m = best[q];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int h = __any_sync(0xffffffffu, have[q]);
        if (lane == 0) {
          red_max[q][warp] = m;
          red_have[q][warp] = h;
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (tid < tq) {
        float m = -INFINITY;
        int h = 0;
        for (int w2 = 0; w2 < kSelThreads / 32; ++w2) {
          m = fmaxf(m, red_max[tid][w2]);
          h |= red_have[tid][w2];
        }
        a.score[((long long)(q0 + tid) * a.Hkv + x.g) * a.max_blocks + b] = h ? m : NAN;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the sums are read before the next unit writes them
    }
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < kShortStages; ++i) {
      mbar_inval(&full[i]);
      mbar_inval(&empty[i]);
    }
}

// k_select_long: a unit's 128 queries x 128 keys of dot products, blocked
// like a matrix product.  The dimensions pass in chunks of 32: each chunk of
// the queries and of the keys is staged in shared memory as FP32, transposed
// ([dimension][query or key]); thread (qg, kg) keeps an 8 x 8 tile of
// accumulators (queries 8 qg .. 8 qg + 7, keys 4 kg .. 4 kg + 3 and
// 64 + 4 kg .. 64 + 4 kg + 3) and adds one FMA per dimension to each, in
// dimension order from +0, so every dot is the reading's exact sum.  Four
// 16-byte shared-memory reads feed 64 FMAs.
constexpr int kLongThreads = 256;
constexpr int kLongChunk = 32;  // dimensions staged at a time
struct LongSmem {
  float q[kLongChunk][128];
  float k[kLongChunk][128];
  int kvis[128];  // key on a valid page inside the sequence
  int qlim[128];  // keys a query sees (0: no query)
};

__host__ __device__ constexpr size_t long_smem(int) { return sizeof(LongSmem); }

// 16 consecutive values from `base` (16-byte aligned), widened to FP32
__device__ __forceinline__ void load16(const uint8_t* base, int dtype, float* out) {
  if (dtype == MXSA_FP8_E4M3) {
    unpack_e4m3x16(__ldg(reinterpret_cast<const uint4*>(base)), out);
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(base);
    unpack_16bitx8(__ldg(p), dtype == MXSA_BF16, out);
    unpack_16bitx8(__ldg(p + 1), dtype == MXSA_BF16, out + 8);
  }
}

template <int D>
__global__ void __launch_bounds__(kLongThreads, 2)
    k_select_long(SelArgs a) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  LongSmem& sm = *reinterpret_cast<LongSmem*>(sm_raw);
  // Let through once every k_select_short CTA has passed its wait for the
  // table, so the table is complete; this launch waits for k_select_short
  // itself only at its end (k_select_topk waits on this launch).
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int Hkv = a.Hkv;
  const int esz = a.dtype == MXSA_FP8_E4M3 ? 1 : 2;
  const int qg = tid >> 4, kg = tid & 15;
  const int row = tid & 127, half = tid >> 7;  // staging: row, 16 dimensions of the chunk
  const long long units = a.tab.unit_long[a.B] * Hkv;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int g = (int)(u % Hkv);
    const long long v = u / Hkv;
    const int s = unit_seq(a.tab.unit_long, a.B, v);
    const SeqRec r = a.tab.seq[s];
    const long long w = v - a.tab.unit_long[s];
    const int b = (int)(w % r.nblk), chunk = (int)(w / r.nblk);
    const int tq = r.tq, L = r.L, q0 = r.q0;
    // this thread's staging rows: key 128 b + row and query chunk * 128 + row
    const int key = 128 * b + row;
    int page = -1;
    if (key < L) {
      page = a.bt[(long long)s * a.max_pages + key / a.ps];
      if (page < 0 || page >= a.num_pages) page = -1;
    }
    const int qi = chunk * 128 + row;
    __syncthreads();  // the previous unit is done with the shared memory
    if (half == 0) {
      sm.kvis[row] = page >= 0;
      int lim = 0;
      if (qi < tq) {
        lim = min(128, L - 128 * b);
        if (a.causal) lim = min(lim, L - tq + qi - 128 * b + 1);
      }
      sm.qlim[row] = lim;
    }
    const uint8_t* krow =
        page >= 0 ? a.ik + ((((long long)page * Hkv + g) * a.ps + key % a.ps) * D) * esz : nullptr;
    const uint8_t* qrow = qi < tq ? a.iq + (((long long)(q0 + qi) * Hkv + g) * D) * esz : nullptr;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 1
    for (int d0 = 0; d0 < D; d0 += kLongChunk) {
      float x[16];
      if (krow) load16(krow + (size_t)(d0 + 16 * half) * esz, a.dtype, x);
      else
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) sm.k[16 * half + j][row] = x[j];
      if (qrow) load16(qrow + (size_t)(d0 + 16 * half) * esz, a.dtype, x);
      else
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) sm.q[16 * half + j][row] = x[j];
      __syncthreads();
#pragma unroll 4
      for (int dl = 0; dl < kLongChunk; ++dl) {
        const float4 qa = *reinterpret_cast<const float4*>(&sm.q[dl][8 * qg]);
        const float4 qb = *reinterpret_cast<const float4*>(&sm.q[dl][8 * qg + 4]);
        const float4 ka = *reinterpret_cast<const float4*>(&sm.k[dl][4 * kg]);
        const float4 kb = *reinterpret_cast<const float4*>(&sm.k[dl][64 + 4 * kg]);
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const float kv[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(qv[i], kv[j], acc[i][j]);
      }
      __syncthreads();  // the chunk is read before the next one is staged
    }
    // block maximum per query over its visible keys (NaN dots skipped),
    // then over the 16 threads that share the query
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int qr = 8 * qg + i;
      const int lim = sm.qlim[qr];
      float m = -INFINITY;
      int h = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int kp = j < 4 ? 4 * kg + j : 64 + 4 * kg + (j - 4);
        const float x = acc[i][j];
        if (kp >= lim || !sm.kvis[kp] || isnan(x)) continue;
        if (!h || x > m) m = x;
        h = 1;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, off);
        const int oh = __shfl_xor_sync(0xffffffffu, h, off);
        if (oh && (!h || om > m)) m = om;
        h |= oh;
      }
      const int qq = chunk * 128 + qr;
      if (kg == 0 && qq < tq) a.score[((long long)(q0 + qq) * Hkv + g) * a.max_blocks + b] = h ? m : NAN;
    }
  }
  pdl_wait();  // leave only after k_select_short has completed
}

// Order-preserving 64-bit key of (score, block): larger = earlier in the
// selection.  -0 ranks as +0; a block without a score gets 0.
__device__ __forceinline__ unsigned long long rank_key(float x, int b) {
  if (x == 0.f) x = 0.f;
  uint32_t u = __float_as_uint(x);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - (uint32_t)b);
}

__global__ void __launch_bounds__(kTopkThreads)
    k_select_topk(SelArgs a) {
  __shared__ unsigned long long key[kSelMaxBlocks];
  pdl_launch_dependents();
  pdl_wait();  // the block scores are complete
  const bool bad = *a.tab.bad != 0;
  const long long rows = (long long)a.total_q * a.Hkv;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int t = (int)(row / a.Hkv);
    int32_t* out = a.sel + row * a.topk;
    int nb = 0;
    if (!bad) {
      int lo = 0, hi = a.B - 1;  // the sequence of token t: the last s with q0 <= t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.tab.seq[mid].q0 <= t) lo = mid;
        else hi = mid - 1;
      }
      const SeqRec r = a.tab.seq[lo];
      if (t >= r.q0 && t < r.q0 + r.tq) nb = r.nblk;
    }
    int n2 = 1;
    while (n2 < nb) n2 <<= 1;
    const float* sc = a.score + row * a.max_blocks;
    __syncthreads();  // the previous row's keys are read
    for (int i = threadIdx.x; i < n2; i += blockDim.x) {
      unsigned long long k = 0;
      if (i < nb) {
        const float x = sc[i];
        if (!isnan(x)) k = rank_key(x, i);
      }
      key[i] = k;
    }
    __syncthreads();
    // bitonic sort, descending
    for (int size = 2; size <= n2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = threadIdx.x; i < n2 / 2; i += blockDim.x) {
          const int lo2 = 2 * i - (i & (stride - 1));
          const int hi2 = lo2 + stride;
          const bool desc = (lo2 & size) == 0;
          const unsigned long long x = key[lo2], y = key[hi2];
          if ((x < y) == desc) {
            key[lo2] = y;
            key[hi2] = x;
          }
        }
        __syncthreads();
      }
    }
    for (int k = threadIdx.x; k < a.topk; k += blockDim.x) {
      const unsigned long long kk = k < n2 ? key[k] : 0ull;
      out[k] = kk ? (int32_t)(0xffffffffu - (uint32_t)(kk & 0xffffffffu)) : -1;
    }
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

// Workspace: the block scores, then the sequence table.
size_t select_score_bytes(const mxsa_problem& p) {
  return (size_t)p.total_q * p.num_kv_heads * (size_t)max_blocks_per_seq(p) * sizeof(float);
}

size_t select_workspace_bytes(const mxsa_problem& p) {
  const size_t B = (size_t)p.num_seqs;
  return align256(select_score_bytes(p)) + align256(B * sizeof(SeqRec)) + 2 * align256((B + 1) * 8) + 256;
}

// 3-D map of the index-key cache [pages * Hkv][page_size][idx_dim] for the
// short scorer: box = one page's rows x one segment of at most 128 bytes,
// 128-byte swizzle (64-byte for the 64-byte rows of FP8 64-dim keys).
static bool make_idx_map(CUtensorMap* m, const void* ik, const mxsa_problem& p, int D) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  if (!fn) return false;
  const bool fp8 = p.kv_dtype == MXSA_FP8_E4M3;
  const cuuint64_t esz = fp8 ? 1 : 2;
  const int span = short_span(D, (int)esz);
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.page_size, (cuuint64_t)p.num_pages * p.num_kv_heads};
  cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)D * esz * p.page_size};
  cuuint32_t box[3] = {(cuuint32_t)(span / esz), (cuuint32_t)(p.page_size == 128 ? 128 : 64), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const CUresult r = fn(m, dt, 3, const_cast<void*>(ik), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_select(const mxsa_problem& p, int idx_dim, const void* iq, const void* ik,
                          const int32_t* bt, const int64_t* cu, const int32_t* lens, void* ws, int32_t* sel,
                          int32_t* flags, cudaStream_t st) {
  if ((long long)p.total_q * p.num_kv_heads == 0) return cudaSuccess;
  SelArgs a;
  a.iq = static_cast<const uint8_t*>(iq);
  a.ik = static_cast<const uint8_t*>(ik);
  a.bt = bt;
  a.cu = cu;
  a.lens = lens;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.score = reinterpret_cast<float*>(w);
  size_t o = align256(select_score_bytes(p));
  a.tab.seq = reinterpret_cast<SeqRec*>(w + o);
  o += align256((size_t)p.num_seqs * sizeof(SeqRec));
  a.tab.unit_short = reinterpret_cast<long long*>(w + o);
  o += align256((size_t)(p.num_seqs + 1) * 8);
  a.tab.unit_long = reinterpret_cast<long long*>(w + o);
  o += align256((size_t)(p.num_seqs + 1) * 8);
  a.tab.bad = reinterpret_cast<int32_t*>(w + o);
  a.sel = sel;
  a.flags = flags;
  a.B = p.num_seqs;
  a.total_q = p.total_q;
  a.Hkv = p.num_kv_heads;
  a.D = idx_dim;
  a.ps = p.page_size;
  a.num_pages = p.num_pages;
  a.max_pages = p.max_pages_per_seq;
  a.max_blocks = (int)max_blocks_per_seq(p);
  a.topk = p.topk;
  a.causal = p.causal;
  a.dtype = p.kv_dtype;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int esz = p.kv_dtype == MXSA_FP8_E4M3 ? 1 : 2;
  static cudaError_t attr_err = [] {
    cudaError_t e = cudaSuccess;
    const void* k[6] = {(const void*)k_select_short<64, false>, (const void*)k_select_short<128, false>,
                        (const void*)k_select_short<64, true>,  (const void*)k_select_short<128, true>,
                        (const void*)k_select_long<64>,         (const void*)k_select_long<128>};
    const size_t bytes[6] = {short_smem(64, 2), short_smem(128, 2), short_smem(64, 1),
                             short_smem(128, 1), long_smem(64),     long_smem(128)};
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
      e = cudaFuncSetAttribute(k[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes[i]);
    return e;
  }();
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tmk;
  if (!make_idx_map(&tmk, ik, p, idx_dim)) return cudaErrorInvalidValue;
  // persistent grids: as many CTAs as fit at once (a second, partial wave
  // would start only when the first finishes)
  auto grid_for = [&](const void* kern, size_t smem, int threads) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    return dim3((unsigned)(sms * per_sm));
  };
  cudaError_t e = launch_pdl(k_select_prep, dim3(1), dim3(kPrepThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  const size_t ss = short_smem(idx_dim, esz), sl = long_smem(idx_dim);
  auto short_kernel = [&](auto kern) {
    return launch_pdl(kern, grid_for((const void*)kern, ss, kShortThreads), dim3(kShortThreads), ss, st, tmk, a);
  };
  const bool fp8 = p.kv_dtype == MXSA_FP8_E4M3;
  if (idx_dim == 64) {
    e = fp8 ? short_kernel(k_select_short<64, true>) : short_kernel(k_select_short<64, false>);
    if (e == cudaSuccess)
      e = launch_pdl(k_select_long<64>, grid_for((const void*)k_select_long<64>, sl, kLongThreads),
                     dim3(kLongThreads), sl, st, a);
  } else {
    e = fp8 ? short_kernel(k_select_short<128, true>) : short_kernel(k_select_short<128, false>);
    if (e == cudaSuccess)
      e = launch_pdl(k_select_long<128>, grid_for((const void*)k_select_long<128>, sl, kLongThreads),
                     dim3(kLongThreads), sl, st, a);
  }
  if (e != cudaSuccess) return e;
  const long long rows = (long long)p.total_q * p.num_kv_heads;
  const long long grid = rows < (long long)sms * 8 ? rows : (long long)sms * 8;
  return launch_pdl(k_select_topk, dim3((unsigned)grid), dim3(kTopkThreads), 0, st, a);
}

}  // namespace mxsa
