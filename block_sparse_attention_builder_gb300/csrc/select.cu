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
// Two launches:
//   k_select_score  persistent CTAs of 128 threads over work units (sequence,
//                   block, kv head, query chunk).  A sequence with at most 8
//                   new tokens: thread p holds key 128 b + p and the block's
//                   maximum per query comes from a CTA reduction (the index
//                   keys are read once, the HBM-bound decode case).  Longer
//                   sequences: the block's keys are staged in shared memory
//                   as FP32 and thread i owns query i of a 128-query chunk,
//                   walking the block's keys itself (no reduction).
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
constexpr int kSelSeqMax = 1024;     // sequences (the per-CTA table)
constexpr int kSelMaxBlocks = 4096;  // blocks per sequence (the sort buffer)
constexpr int kSelSmallTq = 8;       // at most this many new tokens: one thread per key
constexpr int kTopkThreads = 256;

struct SelArgs {
  const uint8_t* iq;        // [total_q][Hkv][D]
  const uint8_t* ik;        // [pages][Hkv][ps][D]
  const int32_t* bt;
  const int64_t* cu;
  const int32_t* lens;
  float* score;             // [total_q][Hkv][max_blocks]
  int32_t* sel;             // [total_q][Hkv][topk]
  int32_t* flags;           // may be null
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

// Per-sequence table every CTA builds for itself: L (clamped), first token,
// new tokens, blocks, and the exclusive prefix of work units.  Returns
// false (uniform) when cu_seqlens_q is not a non-decreasing partition of
// [0, total_q].
struct SeqTable {
  int32_t* L;
  int32_t* q0;
  int32_t* tq;
  int32_t* nblk;
  long long* unit0;  // [B + 1]
};

__device__ bool build_table(const SelArgs& a, SeqTable T, long long* total_units) {
  __shared__ int s_bad;
  __shared__ long long s_part[kSelThreads];
  if (threadIdx.x == 0) s_bad = (a.cu[0] != 0 || a.cu[a.B] != a.total_q) ? 1 : 0;
  __syncthreads();
  const long long cap = (long long)a.max_pages * a.ps;
  // each thread owns a contiguous run of sequences
  const int per = (a.B + kSelThreads - 1) / kSelThreads;
  const int s0 = threadIdx.x * per, s1 = min(a.B, s0 + per);
  long long run = 0;
  for (int s = s0; s < s1; ++s) {
    const long long c0 = a.cu[s], c1 = a.cu[s + 1];
    if (c1 < c0) s_bad = 1;
    long long L = a.lens[s];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int tq = (int)(c1 > c0 ? c1 - c0 : 0);
    const int nb = (int)((L + 127) / 128);
    T.L[s] = (int)L;
    T.q0[s] = (int)c0;
    T.tq[s] = tq;
    T.nblk[s] = nb;
    const int chunks = tq == 0 ? 0 : (tq <= kSelSmallTq ? 1 : (tq + kSelThreads - 1) / kSelThreads);
    run += (long long)nb * chunks;
  }
  s_part[threadIdx.x] = run;
  __syncthreads();
  if (threadIdx.x == 0) {  // few values: a serial scan is enough
    long long acc = 0;
    for (int i = 0; i < kSelThreads; ++i) {
      const long long v = s_part[i];
      s_part[i] = acc;
      acc += v;
    }
    *total_units = acc;
  }
  __syncthreads();
  long long u = s_part[threadIdx.x];
  for (int s = s0; s < s1; ++s) {
    T.unit0[s] = u;
    const int tq = T.tq[s];
    const int chunks = tq == 0 ? 0 : (tq <= kSelSmallTq ? 1 : (tq + kSelThreads - 1) / kSelThreads);
    u += (long long)T.nblk[s] * chunks;
  }
  if (threadIdx.x == kSelThreads - 1) T.unit0[a.B] = *total_units;
  __syncthreads();
  return s_bad == 0;
}

template <int D>
__global__ void __launch_bounds__(kSelThreads)
    k_select_score(SelArgs a) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  __shared__ int32_t tL[kSelSeqMax], tq0[kSelSeqMax], ttq[kSelSeqMax], tnb[kSelSeqMax];
  __shared__ long long tu0[kSelSeqMax + 1];
  __shared__ long long s_total;
  __shared__ float red_max[kSelSmallTq][kSelThreads / 32];
  __shared__ int red_have[kSelSmallTq][kSelThreads / 32];
  pdl_launch_dependents();
  pdl_wait();
  const SeqTable T{tL, tq0, ttq, tnb, tu0};
  if (!build_table(a, T, &s_total)) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.flags) atomicOr(a.flags, MXSA_FLAG_CU);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = a.Hkv;
  float* kf = reinterpret_cast<float*>(sm_raw);              // [128][D] keys (long sequences)
  float* qs = kf;                                             // [8][D] queries (short sequences)
  int* kvis = reinterpret_cast<int*>(kf + kSelThreads * D);  // [128]: key p visible (length, page)
  const long long units = s_total * Hkv;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int g = (int)(u % Hkv);
    const long long v = u / Hkv;
    int lo = 0, hi = a.B - 1;  // last s with unit0[s] <= v
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tu0[mid] <= v) lo = mid;
      else hi = mid - 1;
    }
    const int s = lo;
    const int nb = tnb[s], tq = ttq[s], L = tL[s], q0 = tq0[s];
    const long long w = v - tu0[s];
    const int b = (int)(w % nb), chunk = (int)(w / nb);
    // this thread's key position and whether it is on a valid page
    const int p = 128 * b + tid;
    int page = -1;
    if (p < L) {
      page = a.bt[(long long)s * a.max_pages + p / a.ps];
      if (page < 0 || page >= a.num_pages) page = -1;
    }
    const long long kbase = (((long long)(page < 0 ? 0 : page) * Hkv + g) * a.ps + p % a.ps) * D;
    if (tq <= kSelSmallTq) {
      // ---- one thread per key; the block maximum of each query by reduction
      __syncthreads();  // the previous unit's shared memory is free
      for (int i = tid; i < tq * D; i += kSelThreads)
        qs[i] = elem(a.iq, ((long long)(q0 + i / D) * Hkv + g) * D + i % D, a.dtype);
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
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
          const float kd = elem(a.ik, kbase + d, a.dtype);
#pragma unroll
          for (int i = 0; i < kSelSmallTq; ++i)
            if (i < tq) acc[i] = __fmaf_rn(qs[i * D + d], kd, acc[i]);
        }
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
    } else {
      // ---- one thread per query of the chunk; the block's keys in shared
      // memory as FP32 (exact widening), with their visibility
      __syncthreads();
      for (int i = tid; i < kSelThreads * D; i += kSelThreads) {
        const int pp = i / D, d = i % D;
        const int key = 128 * b + pp;
        float x = 0.f;
        if (key < L) {
          const int pg = a.bt[(long long)s * a.max_pages + key / a.ps];
          if (pg >= 0 && pg < a.num_pages) x = elem(a.ik, (((long long)pg * Hkv + g) * a.ps + key % a.ps) * D + d, a.dtype);
        }
        kf[i] = x;
      }
      kvis[tid] = page >= 0 ? 1 : 0;
      __syncthreads();
      const int i = chunk * kSelThreads + tid;  // this thread's query of the sequence
      if (i < tq) {
        float q[D];
        const long long qb = ((long long)(q0 + i) * Hkv + g) * D;
#pragma unroll
        for (int d = 0; d < D; ++d) q[d] = elem(a.iq, qb + d, a.dtype);
        const int pos = L - tq + i;
        int lim = min(128, L - 128 * b);
        if (a.causal) lim = min(lim, pos - 128 * b + 1);
        float m = -INFINITY;
        int h = 0;
        for (int pp = 0; pp < lim; ++pp) {
          if (!kvis[pp]) continue;
          const float* kr = kf + pp * D;
          float acc = 0.f;
#pragma unroll
          for (int d = 0; d < D; ++d) acc = __fmaf_rn(q[d], kr[d], acc);
          if (isnan(acc)) continue;
          if (!h || acc > m) m = acc;
          h = 1;
        }
        a.score[((long long)(q0 + i) * Hkv + g) * a.max_blocks + b] = h ? m : NAN;
      }
    }
  }
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
  __shared__ int s_bad;
  pdl_launch_dependents();
  pdl_wait();  // the block scores are complete
  if (threadIdx.x == 0) s_bad = (a.cu[0] != 0 || a.cu[a.B] != a.total_q) ? 1 : 0;
  __syncthreads();
  for (int s = threadIdx.x; s < a.B; s += blockDim.x)
    if (a.cu[s + 1] < a.cu[s]) s_bad = 1;
  __syncthreads();
  const bool bad = s_bad != 0;
  const long long rows = (long long)a.total_q * a.Hkv;
  const long long cap = (long long)a.max_pages * a.ps;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int t = (int)(row / a.Hkv);
    int32_t* out = a.sel + row * a.topk;
    int nb = 0;
    if (!bad) {
      int lo = 0, hi = a.B - 1;  // the sequence of token t: last s with cu[s] <= t ...
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      while (lo < a.B - 1 && a.cu[lo + 1] <= t) ++lo;  // ... skipping empty sequences
      long long L = a.lens[lo];
      L = L < 0 ? 0 : (L > cap ? cap : L);
      if (t >= a.cu[lo] && t < a.cu[lo + 1]) nb = (int)((L + 127) / 128);
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
  if (bad && blockIdx.x == 0 && threadIdx.x == 0 && a.flags) atomicOr(a.flags, MXSA_FLAG_CU);
}

}  // namespace

size_t select_score_bytes(const mxsa_problem& p) {
  return (size_t)p.total_q * p.num_kv_heads * (size_t)max_blocks_per_seq(p) * sizeof(float);
}

cudaError_t launch_select(const mxsa_problem& p, int idx_dim, const void* iq, const void* ik,
                          const int32_t* bt, const int64_t* cu, const int32_t* lens, float* score, int32_t* sel,
                          int32_t* flags, cudaStream_t st) {
  if ((long long)p.total_q * p.num_kv_heads == 0) return cudaSuccess;
  SelArgs a;
  a.iq = static_cast<const uint8_t*>(iq);
  a.ik = static_cast<const uint8_t*>(ik);
  a.bt = bt;
  a.cu = cu;
  a.lens = lens;
  a.score = score;
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
  const size_t smem = (size_t)kSelThreads * idx_dim * sizeof(float) + kSelThreads * sizeof(int);
  static cudaError_t attr_err = [] {
    const int bytes = (int)((size_t)kSelThreads * 128 * sizeof(float) + kSelThreads * sizeof(int));
    cudaError_t e = cudaFuncSetAttribute(k_select_score<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_select_score<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
  }();
  if (attr_err != cudaSuccess) return attr_err;
  cudaError_t e = idx_dim == 64 ? launch_pdl(k_select_score<64>, dim3(sms * 4), dim3(kSelThreads), smem, st, a)
                                : launch_pdl(k_select_score<128>, dim3(sms * 4), dim3(kSelThreads), smem, st, a);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)p.total_q * p.num_kv_heads;
  const long long grid = rows < (long long)sms * 8 ? rows : (long long)sms * 8;
  return launch_pdl(k_select_topk, dim3((unsigned)grid), dim3(kTopkThreads), 0, st, a);
}

}  // namespace mxsa
