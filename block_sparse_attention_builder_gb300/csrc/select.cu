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
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>

#include "internal.h"

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

__device__ __forceinline__ float elem(const uint8_t* base, int64_t i, int dtype) {
  if (dtype == MXSA_FP8_E4M3) {
    const uint16_t two = base[i];
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
  }
  const uint16_t bits = reinterpret_cast<const uint16_t*>(base)[i];
  if (dtype == MXSA_BF16) return __uint_as_float((uint32_t)bits << 16);
  return __half2float(__ushort_as_half(bits));
}

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

// Dot products of one staged key row with the first tq (<= NQ) queries,
// each summed by fused multiply-adds in dimension order.
template <int NQ, int D>
__device__ __forceinline__ void short_dots(const uint8_t* row, const float* qs, int dtype, float* acc, int tq = NQ) {
  if (dtype == MXSA_FP8_E4M3) {
#pragma unroll 2
    for (int cc = 0; cc < D / 16; ++cc) {
      float kd[16];
      unpack_e4m3x16(*reinterpret_cast<const uint4*>(row + cc * 16), kd);
#pragma unroll
      for (int e = 0; e < 16; ++e)
#pragma unroll
        for (int i = 0; i < NQ; ++i)
          if (i < tq) acc[i] = __fmaf_rn(qs[i * D + cc * 16 + e], kd[e], acc[i]);
    }
  } else {
    const bool bf16 = dtype == MXSA_BF16;
#pragma unroll 2
    for (int cc = 0; cc < D / 8; ++cc) {
      float kd[8];
      unpack_16bitx8(*reinterpret_cast<const uint4*>(row + cc * 16), bf16, kd);
#pragma unroll
      for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int i = 0; i < NQ; ++i)
          if (i < tq) acc[i] = __fmaf_rn(qs[i * D + cc * 8 + e], kd[e], acc[i]);
    }
  }
}

// shared memory of k_select_short: 8 FP32 queries, then 128 raw key rows
// padded by 16 bytes (each thread reads its own row without bank conflicts)
__host__ __device__ constexpr size_t short_smem(int D, int esz) {
  return (size_t)kSelSmallTq * D * sizeof(float) + (size_t)kSelThreads * (D * esz + 16);
}

template <int D>
__global__ void __launch_bounds__(kSelThreads)
    k_select_short(SelArgs a) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  __shared__ float red_max[kSelSmallTq][kSelThreads / 32];
  __shared__ int red_have[kSelSmallTq][kSelThreads / 32];
  pdl_wait();  // the sequence table
  // only now: k_select_long reads the table without a wait of its own
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = a.Hkv;
  const int esz = a.dtype == MXSA_FP8_E4M3 ? 1 : 2;
  const int row_bytes = D * esz + 16;
  float* qs = reinterpret_cast<float*>(sm_raw);                      // [8][D]
  uint8_t* kst = sm_raw + kSelSmallTq * D * sizeof(float);           // [128][row_bytes]
  const long long units = a.tab.unit_short[a.B] * Hkv;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int g = (int)(u % Hkv);
    const long long v = u / Hkv;
    const int s = unit_seq(a.tab.unit_short, a.B, v);
    const SeqRec r = a.tab.seq[s];
    const int b = (int)(v - a.tab.unit_short[s]);
    const int tq = r.tq, L = r.L, q0 = r.q0;
    // this thread's key position and whether it is on a valid page
    const int p = 128 * b + tid;
    int page = -1;
    if (p < L) {
      page = a.bt[(long long)s * a.max_pages + p / a.ps];
      if (page < 0 || page >= a.num_pages) page = -1;
    }
    __syncthreads();  // the previous unit's shared memory is free
    for (int i = tid; i < tq * D; i += kSelThreads)
      qs[i] = elem(a.iq, ((long long)(q0 + i / D) * Hkv + g) * D + i % D, a.dtype);
    // the block's pages (one for 128-token pages, two for 64), read once;
    // then every 16-byte chunk of the thread's share issued before any is
    // stored, so the copies overlap (consecutive threads: consecutive
    // chunks of a row)
    const int chunks_row = D * esz / 16;  // 16-byte chunks per key row: 4, 8 or 16
    int pg_lo = -1, pg_hi = -1;  // the pages of rows 0-63 and 64-127
    if (128 * b < L) {
      const int pg = a.bt[(long long)s * a.max_pages + (128 * b) / a.ps];
      pg_lo = (pg >= 0 && pg < a.num_pages) ? pg : -1;
    }
    if (a.ps == 128) {
      pg_hi = pg_lo;
    } else if (128 * b + 64 < L) {
      const int pg = a.bt[(long long)s * a.max_pages + (128 * b + 64) / a.ps];
      pg_hi = (pg >= 0 && pg < a.num_pages) ? pg : -1;
    }
    uint4 xs[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i >= chunks_row) break;
      const int c = i * kSelThreads + tid;
      const int rr = c / chunks_row, cc = c % chunks_row;
      const int key = 128 * b + rr;
      const int pg = rr < 64 ? pg_lo : pg_hi;
      xs[i] = make_uint4(0, 0, 0, 0);
      if (key < L && pg >= 0)
        xs[i] = __ldcs(reinterpret_cast<const uint4*>(
                           a.ik + ((((long long)pg * Hkv + g) * a.ps + key % a.ps) * D) * esz) +
                       cc);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i >= chunks_row) break;
      const int c = i * kSelThreads + tid;
      const int rr = c / chunks_row, cc = c % chunks_row;
      *reinterpret_cast<uint4*>(kst + rr * row_bytes + cc * 16) = xs[i];
    }
    __syncthreads();
    float best[kSelSmallTq];
    int have[kSelSmallTq];
#pragma unroll
    for (int i = 0; i < kSelSmallTq; ++i) {
      best[i] = -INFINITY;
      have[i] = 0;
    }
    if (page >= 0) {
      float acc[kSelSmallTq];
#pragma unroll
      for (int i = 0; i < kSelSmallTq; ++i) acc[i] = 0.f;
      const uint8_t* row = kst + tid * row_bytes;
      if (tq == 1)
        short_dots<1, D>(row, qs, a.dtype, acc);
      else
        short_dots<kSelSmallTq, D>(row, qs, a.dtype, acc, tq);
#pragma unroll
      for (int i = 0; i < kSelSmallTq; ++i) {
        const int pos = L - tq + i;
        const bool vis = i < tq && (!a.causal || p <= pos) && !isnan(acc[i]);
        if (vis) {
          best[i] = acc[i];
          have[i] = 1;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kSelSmallTq; ++i) {
      if (i >= tq) break;
      float m = best[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int h = __any_sync(0xffffffffu, have[i]);
      if (lane == 0) {
        red_max[i][warp] = m;
        red_have[i][warp] = h;
      }
    }
    __syncthreads();
    if (tid < tq) {
      float m = -INFINITY;
      int h = 0;
      for (int w2 = 0; w2 < kSelThreads / 32; ++w2) {
        m = fmaxf(m, red_max[tid][w2]);
        h |= red_have[tid][w2];
      }
      a.score[((long long)(q0 + tid) * Hkv + g) * a.max_blocks + b] = h ? m : NAN;
    }
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
    const void* k[4] = {(const void*)k_select_short<64>, (const void*)k_select_short<128>,
                        (const void*)k_select_long<64>, (const void*)k_select_long<128>};
    const size_t bytes[4] = {short_smem(64, 2), short_smem(128, 2), long_smem(64), long_smem(128)};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = cudaFuncSetAttribute(k[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes[i]);
    return e;
  }();
  if (attr_err != cudaSuccess) return attr_err;
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
  if (idx_dim == 64) {
    e = launch_pdl(k_select_short<64>, grid_for((const void*)k_select_short<64>, ss, kSelThreads), dim3(kSelThreads),
                   ss, st, a);
    if (e == cudaSuccess)
      e = launch_pdl(k_select_long<64>, grid_for((const void*)k_select_long<64>, sl, kLongThreads),
                     dim3(kLongThreads), sl, st, a);
  } else {
    e = launch_pdl(k_select_short<128>, grid_for((const void*)k_select_short<128>, ss, kSelThreads),
                   dim3(kSelThreads), ss, st, a);
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
