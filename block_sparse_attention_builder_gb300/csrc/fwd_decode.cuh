// KV-outer forward for decode work items (fw-ai/minimax-kernels README,
// intro: a selected KV block is loaded once for the queries that selected
// it).  In a sequence with one new token every selected block of a KV head
// is selected by that one token, so the scheduler hands this kernel runs of
// up to 8 such blocks; each block is still loaded from HBM exactly once,
// and the run's partial results are merged on chip by an online softmax,
// leaving one partial (o, lse) per run instead of one per block.
//
// With only G (<= 16) query rows per block, the products are computed
// transposed so that the 128 keys fill the MMA's M dimension:
//   S^T = K Q^T   (M = 128 keys, N = rows padded to 16, K = 128)
//   O^T += V^T P^T (M = 128 head dims, N = rows, K = 128 keys)
// Accumulators live in tensor memory; softmax thread k owns key k of S^T
// and head dim k of O^T.  The row maximum m is only raised when a block's
// score exceeds it by more than 2^8 (then O^T and the per-thread sums are
// rescaled), so most blocks need no cross-thread reduction.
//
// The decode phase of the forward kernel (fwd.cu), run by each CTA on its
// decode items before its KV-stationary items: warps 0-3 softmax/epilogue,
// warp 4 TMA producer (q rows of the item; K and V pages of each block into
// a 3-stage ring; FP8 / NVFP4 rows into the V half of the block's stage),
// warp 5 issues the S^T MMAs and warp 10 the O^T MMAs, warps 6-9 widen (FP8
// / NVFP4: each block's narrow rows into the q dtype, in place); the
// kernel's other warps idle through this phase.  TMEM columns [0, 64) of
// the CTA's allocation hold S^T and O^T.
#pragma once
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

namespace dec {

constexpr uint32_t kKVTile = 32768;  // 128 keys x 128 x 16-bit
constexpr uint32_t kStage = 2 * kKVTile;
constexpr int kMaxStages = 3;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct BlockInfo {
  int32_t valid, pad0, pad1, pad2;
};

struct Ctrl {
  uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], p_empty[2], o_full[2], o_empty[2];
  // widened caches: stg_full[st], the block's narrow rows landed in stage st
  uint64_t stg_full[kMaxStages], done;
  uint32_t tmem_base;
  int32_t abort_flag;
  BlockInfo info[kMaxStages];
  float inv_l[2][16];    // 1 / l per row of an item whose epilogue is pending, by O buffer
  float lse[2][16];      // and its lse per row
};

// cache kinds, the forward's template parameter: 16-bit (the q dtype), and
// the two that are staged and widened, FP8 and NVFP4
constexpr int kKv16 = kKind16, kKvFp8 = kKindFp8, kKvFp4 = kKindFp4;

struct DecArgs {
  const int32_t* block_tables;
  const SeqInfo* seq;
  const int32_t* active;
  const int32_t* row_ptr;
  const int4* items;
  const int32_t* cta_ptr;
  const int32_t* idx_hdr;
  const int32_t* sch_hdr;
  void* part_o;  // partial rows: FP32 when part32, else the 16-bit q dtype
  float* part_lse;
  int32_t* flags;
  // kv_fp8: blocks are staged and widened (FP8 or NVFP4); kv_fp4: NVFP4,
  // whose scale rows come from kbase / vbase by bulk copies
  int32_t num_seqs, Hq, Hkv, G, page_size, max_pages, num_pages, kv_fp8, ab_bf16, ns, part32, kv_fp4;
  const uint8_t* kbase;
  const uint8_t* vbase;
  float scale_log2;
};

struct Layout {
  uint32_t q, p, red, ctrl, total;
};

// Widened caches need no room of their own: a block's narrow rows land in
// the V half of its own stage and are widened in place.
template <int N>
__host__ __device__ constexpr Layout smem_layout(int ns) {
  Layout L{};
  L.q = (uint32_t)ns * kStage;
  L.p = L.q + 2u * N * 256u;
  L.red = L.p + 2u * N * 256u;
  L.ctrl = L.red + 4u * N * 4u;
  L.total = L.ctrl + (uint32_t)sizeof(Ctrl);
  return L;
}

template <int N>
constexpr int stages_for(int fp8) {
  (void)fp8;  // widened caches widen in their stage: the same ring
  return N <= 32 ? 3 : 2;
}

// One item's look-ups as the producer warp holds them: uniform fields, and
// per lane j < nk the valid keys, physical pages and entry of block j.
struct BlockDesc {
  int nk, g, row0, valid, page0, page1, entry;
};

// Largest s with seq[s].blk_off <= r, found by the whole warp: each round
// probes 32 evenly spaced sequences, so a batch of up to 1024 sequences
// takes two dependent reads.
__device__ __forceinline__ int warp_seq_of_block(const SeqInfo* seq, int B, int r, int lane) {
  int lo = 0, hi = B;  // seq[lo].blk_off <= r always holds (blk_off[0] = 0)
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = idx < hi && seq[idx].blk_off <= r;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int last = m ? 31 - __clz((int)m) : 0;
    lo += last * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

__device__ __forceinline__ uint32_t swz_kv(uint32_t row, uint32_t chunk16) {
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

__device__ __forceinline__ uint32_t widen_e4m3x2(uint16_t v, int bf16) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  if (!bf16) return h2;
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(h);
  return pack2(f.x, f.y, 1);
}

// NVFP4 rows (E2M1 codes, one E4M3 scale per 16 elements) widened to the
// q dtype: every code times its scale is exact in FP16 (|values| within
// [2^-10, 2688]) and in BF16.  One 32-element chunk c4 of row `row` of a
// [128][128] tile at `dst` (the swz_kv layout) from its 16 code bytes and
// the row's 8 scale bytes.
__device__ __forceinline__ void widen_fp4_chunk(uint4 raw, uint2 sc, uint32_t dst, int row, int c4, int bf16) {
  const uint32_t sw = ((c4 < 2 ? sc.x : sc.y) >> (16 * (c4 & 1))) & 0xFFFFu;
  uint32_t s2[2];
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const uint16_t b = (uint16_t)((sw >> (8 * gi)) & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2[gi]) : "h"((uint16_t)(b | (b << 8))));
  }
  const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(words[w]));
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h[i]), *reinterpret_cast<const __half2*>(&s2[w >> 1]));
      if (bf16) {
        const float2 f = __half22float2(v);
        o[i] = pack2(f.x, f.y, 1);
      } else {
        o[i] = *reinterpret_cast<uint32_t*>(&v);
      }
    }
    st_shared_v4(dst + swz_kv(row, 4 * c4 + w), o[0], o[1], o[2], o[3]);
  }
}

// A whole row from its 64 code bytes and 8 scale bytes in shared memory
// (shared addresses `codes`, `scales`), the chunks in an order rotated by
// the row to spread the code reads over the banks.
__device__ __forceinline__ void widen_fp4_row(uint32_t codes, uint32_t scales, uint32_t dst, int row, int bf16) {
  const uint2 sc = ld_shared_v2(scales);
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    const int c4 = (cc + row) & 3;
    widen_fp4_chunk(ld_shared_v4(codes + c4 * 16), sc, dst, row, c4, bf16);
  }
}

// named barrier 2 over the 128 widening threads (warps 6-9), and the same
// barrier as an and-vote
__device__ __forceinline__ void widen_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ bool widen_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// named barrier 1 over the 128 softmax threads
__device__ __forceinline__ void wg_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool wg_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool wg_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float* v) {
  if constexpr (N == 16) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_ld32(taddr + c * 32, v + c * 32);
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float* v) {
#pragma unroll
  for (int c = 0; c < N / 16; ++c) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[c * 16 + i]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr + c * 16),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// per-row maximum / sum over the 128 softmax threads (result in every thread)
template <int N, bool kMax>
__device__ __forceinline__ void wg_reduce(float* v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < N; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float x = __shfl_xor_sync(0xffffffffu, v[r], o);
      v[r] = kMax ? fmaxf(v[r], x) : v[r] + x;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < N; ++r) red[warp * N + r] = v[r];
  }
  wg_sync();
#pragma unroll
  for (int r = 0; r < N; ++r) {
    const float a = red[r], b = red[N + r], c = red[2 * N + r], d = red[3 * N + r];
    v[r] = kMax ? fmaxf(fmaxf(a, b), fmaxf(c, d)) : (a + b) + (c + d);
  }
  wg_sync();
}

// Runs the CTA's decode items (called by all of the kernel's threads, with
// 1024-aligned shared memory `sm` and the CTA's TMEM base `tmem`).  On
// return every copy and MMA of the phase has completed and its mbarriers are
// invalidated, so the shared memory is free for the next phase.
template <int N, int kKV>
__device__ __forceinline__ void decode_body(const CUtensorMap& tmk, const CUtensorMap& tmv, const CUtensorMap& tmq,
                                            const DecArgs& a, uint8_t* sm, uint32_t tmem) {
  constexpr bool kPart32 = kind_partials_fp32(kKV);
  const Layout L = smem_layout<N>(a.ns);
  Ctrl& c = *reinterpret_cast<Ctrl*>(sm + L.ctrl);
  float* red = reinterpret_cast<float*>(sm + L.red);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns = a.ns;
  const int it_begin = a.cta_ptr[blockIdx.x], it_end = a.cta_ptr[blockIdx.x + 1];
  if (it_begin >= it_end) return;  // uniform: nothing to do

  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&c.kv_full[i], a.kv_fp8 ? 128 : 1);
      mbar_init(&c.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c.q_full[i], 1);
      mbar_init(&c.q_empty[i], 1);
      mbar_init(&c.s_full[i], 1);
      mbar_init(&c.p_full[i], 128);
      mbar_init(&c.p_empty[i], 1);
      mbar_init(&c.o_full[i], 1);
      mbar_init(&c.o_empty[i], 128);
    }
    for (int i = 0; i < ns; ++i) mbar_init(&c.stg_full[i], 1);
    mbar_init(&c.done, 2);  // one commit from each MMA issuer
    c.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &c.abort_flag;
  const uint32_t sbase = smem_u32(sm);
  const int NB = a.idx_hdr[kHdrNB];

  if (warp == 4) {
    // ------------------------------------------------------- producer warp
    // The whole warp looks an item's blocks up one item ahead (lane j:
    // block j), so the dependent index reads (key, sequence, block table)
    // never sit between a stage becoming free and its copy; lane 0 issues
    // the TMA copies.
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      tma_prefetch_desc(&tmq);
    }
    const int ps = a.page_size;
    const int npg = ps == 128 ? 1 : 2;
    const int G = a.G;
    auto lookup = [&](int it) -> BlockDesc {
      BlockDesc d;
      const int4 itm = a.items[it];
      d.nk = itm.w;
      const int key = lane < itm.w ? a.active[itm.x + lane] : 0;
      const int key0 = __shfl_sync(0xffffffffu, key, 0);
      d.g = key0 / NB;
      const int s = warp_seq_of_block(a.seq, a.num_seqs, key0 - d.g * NB, lane);
      const SeqInfo si = a.seq[s];
      d.row0 = si.q_begin * a.Hq + d.g * G;  // q rows t*Hq + g*G .. + N (past G: padding)
      d.valid = 0;
      d.page0 = -1;
      d.page1 = -1;
      d.entry = -1;
      if (lane < itm.w) {
        const int b = key - d.g * NB - si.blk_off;
        d.valid = min(128, si.L - 128 * b);
        for (int pg = 0; pg < npg; ++pg) {
          if (pg * 64 >= d.valid) continue;
          const int lp = ps == 128 ? b : 2 * b + pg;
          const int phys = a.block_tables[(size_t)s * a.max_pages + lp];
          if (phys < 0 || phys >= a.num_pages) {
            atomicOr(a.flags, MXSA_FLAG_PAGE);
            continue;
          }
          if (pg == 0) d.page0 = phys;
          else d.page1 = phys;
        }
        if (lane > 0) d.entry = a.row_ptr[key];
      }
      return d;
    };
    BlockDesc cur = lookup(it_begin);
    int blk = 0, n_it = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
      const int ib = n_it & 1, ui = n_it >> 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&c.q_empty[ib], (ui & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
      if (!ok) break;
      if (lane == 0) {
        uint8_t* qdst = sm + L.q + ib * (N * 256);
        mbar_arrive_expect_tx(&c.q_full[ib], (uint32_t)N * 256u);
        tma_load_2d(qdst, &tmq, &c.q_full[ib], 0, cur.row0);
        tma_load_2d(qdst + N * 128, &tmq, &c.q_full[ib], 64, cur.row0);
      }
      BlockDesc nxt = cur;
      for (int j = 0; j < cur.nk && ok; ++j, ++blk) {
        const int st = blk % ns, us = blk / ns;
        // block blk lands in stage st once the stage's previous block was
        // consumed (its p v); widened caches land their narrow rows in the
        // stage's V half, where the widening warps widen them in place
        ok = __all_sync(0xffffffffu, mbar_wait(&c.kv_empty[st], (us & 1) ^ 1, abort_flag, a.flags,
                                               MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        const int valid = __shfl_sync(0xffffffffu, cur.valid, j);
        const int pg0 = __shfl_sync(0xffffffffu, cur.page0, j);
        const int pg1 = __shfl_sync(0xffffffffu, cur.page1, j);
        if (lane == 0) {
          c.info[st].valid = valid;  // read after kv_full (softmax) or stg_full (widening)
          const int pages[2] = {pg0, pg1};
          const int present = (pg0 >= 0) + (pg1 >= 0);
          uint8_t* kdst = sm + st * kStage;
          uint8_t* vdst = kdst + kKVTile;
          if (!a.kv_fp8) {
            mbar_arrive_expect_tx(&c.kv_full[st], (uint32_t)present * (uint32_t)ps * 512u);
            for (int pg = 0; pg < npg; ++pg) {
              if (pages[pg] < 0) continue;
              const int z = pages[pg] * a.Hkv + cur.g;
              for (int h = 0; h < 2; ++h) {
                tma_load_3d(kdst + h * 16384 + pg * 8192, &tmk, &c.kv_full[st], h * 64, 0, z);
                tma_load_3d(vdst + h * 16384 + pg * 8192, &tmv, &c.kv_full[st], h * 64, 0, z);
              }
            }
          } else if (a.kv_fp4) {
            // NVFP4: code rows by TMA, scale rows by bulk copy; K at 0 and
            // V at 16 KB of the V half (codes, then scales at 8 KB)
            uint64_t* sf = &c.stg_full[st];
            mbar_arrive_expect_tx(sf, (uint32_t)present * (uint32_t)ps * 144u);
            for (int pg = 0; pg < npg; ++pg) {
              if (pages[pg] < 0) continue;
              const int z = pages[pg] * a.Hkv + cur.g;
              const size_t so = (size_t)z * ps * 72 + (size_t)ps * 64;
              tma_load_3d(vdst + pg * ps * 64, &tmk, sf, 0, 0, z);
              tma_load_3d(vdst + 16384 + pg * ps * 64, &tmv, sf, 0, 0, z);
              bulk_load(vdst + 8192 + pg * ps * 8, a.kbase + so, (uint32_t)ps * 8u, sf);
              bulk_load(vdst + 16384 + 8192 + pg * ps * 8, a.vbase + so, (uint32_t)ps * 8u, sf);
            }
          } else {
            // FP8: e4m3 rows of 128 bytes, K at 0 and V at 16 KB of the V half
            uint64_t* sf = &c.stg_full[st];
            mbar_arrive_expect_tx(sf, (uint32_t)present * (uint32_t)ps * 256u);
            for (int pg = 0; pg < npg; ++pg) {
              if (pages[pg] < 0) continue;
              const int z = pages[pg] * a.Hkv + cur.g;
              tma_load_3d(vdst + pg * 8192, &tmk, sf, 0, 0, z);
              tma_load_3d(vdst + 16384 + pg * 8192, &tmv, sf, 0, 0, z);
            }
          }
        }
        if (j == 0) {
          // the next item's look-ups overlap this item's copies
          if (it + 1 < it_end) nxt = lookup(it + 1);
          // the other keys of this run carry no weight of their own (the
          // run's merged partial sits at its first entry)
          if (cur.entry >= 0)
            for (int r = 0; r < G; ++r) a.part_lse[(size_t)cur.entry * G + r] = -INFINITY;
        }
      }
      cur = nxt;
    }
    if (lane == 0) {
      // drain the loads in flight before the CTA may exit
      for (int k = std::max(0, blk - ns); k < blk; ++k)
        mbar_drain(a.kv_fp8 ? &c.stg_full[k % ns] : &c.kv_full[k % ns], (k / ns) & 1, a.flags, MXSA_FLAG_TIMEOUT,
                   kWaitLimitNs);
      if (n_it > 0)
        mbar_drain(&c.q_full[(n_it - 1) & 1], ((n_it - 1) >> 1) & 1, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
    }
  } else if (warp == 5 || warp == 10) {
    // ---------------------------------------------------------- MMA issuers
    // Warp 5 issues S^T = K Q^T of each block, warp 10 O^T += V^T P^T (one
    // thread each, blocking waits on exactly the barriers it needs): issuing
    // one block's eight MMAs takes hundreds of cycles, and with two issuers
    // neither waits behind the other's issue.  S^T of block b needs its K,
    // at an item start its q, and the S buffer it reuses read out (P of
    // block b - 2 written).  P V of block b needs its P, and at an item
    // start the O buffer it reuses read out; it never waits for the next
    // block's load, so a stage is released as soon as its block is consumed.
    if (lane == 0) {
      const bool qk = warp == 5;
      const uint32_t id = idesc_f16(128, N, (uint32_t)a.ab_bf16, qk ? 0 : 1, 0);
      int b = 0, n_it = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
        const int nk = a.items[it].w;
        const int ib = n_it & 1;
        for (int j = 0; j < nk; ++j, ++b) {
          const int st = b % ns, sb = b & 1;
          if (qk) {
            if (j == 0)
              ok = mbar_wait(&c.q_full[ib], (n_it >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            ok = ok && mbar_wait(&c.kv_full[st], (b / ns) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            ok = ok && (b < 2 || mbar_wait(&c.p_full[sb], ((b - 2) >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT,
                                           kWaitLimitNs));
            if (!ok) break;
            tc_fence_after();
            const uint32_t k_s = sbase + st * kStage;
            const uint32_t q_s = sbase + L.q + ib * (N * 256);
            const uint32_t tS = tmem + sb * N;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off_k = (ks >> 2) * 16384u + (ks & 3) * 32u;
              const uint32_t off_q = (ks >> 2) * (uint32_t)(N * 128) + (ks & 3) * 32u;
              mma_f16_ss(tS, smem_desc_sw128(k_s + off_k, 0, 1024), smem_desc_sw128(q_s + off_q, 0, 1024), id,
                         ks > 0);
            }
            mma_commit(&c.s_full[sb]);
            if (j == nk - 1) mma_commit(&c.q_empty[ib]);
          } else {
            ok = mbar_wait(&c.p_full[sb], (b >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
            if (j == 0)
              ok = ok && mbar_wait(&c.o_empty[ib], ((n_it >> 1) & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT,
                                   kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            const uint32_t v_s = sbase + st * kStage + kKVTile;
            const uint32_t p_s = sbase + L.p + sb * (N * 256);
            const uint32_t tO = tmem + 2 * N + ib * N;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off_p = (ks >> 2) * (uint32_t)(N * 128) + (ks & 3) * 32u;
              mma_f16_ss(tO, smem_desc_sw128(v_s + ks * 2048u, 16384, 1024), smem_desc_sw128(p_s + off_p, 0, 1024),
                         id, (j > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(&c.p_empty[sb]);
            mma_commit(&c.kv_empty[st]);
            if (j == nk - 1) mma_commit(&c.o_full[ib]);
          }
        }
      }
      // both issuers' MMAs complete before the CTA moves on (c.done takes
      // one commit from each)
      mma_commit(&c.done);
      mbar_drain(&c.done, 0, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
    }
  } else if (kKV != kKv16 && warp >= 6 && warp < 10) {
    // ------------------------------------------------------ widening warps
    // Widened caches (FP8, NVFP4): thread k turns row k of each block's K
    // and V into the q dtype, zero past the valid keys, while the softmax
    // warps work on the previous block.  The narrow rows sit in the V half
    // of the block's own stage (K rows at 0, V rows at 16 KB).  K widens
    // into the K half.  V widens over itself: widened V row k covers bytes
    // k * 128 of both 16 KB halves of the V half.  For FP8 those are e4m3 K
    // row k (already widened) and e4m3 V row k (read whole first), so each
    // thread only touches its own row.  NVFP4 rows are 64 code bytes and 8
    // scale bytes, so a widened row covers other rows' codes and scales:
    // every thread reads its V row first, and the 128 threads meet at a
    // named barrier before any V byte is written.
    const int k = tid - 192;
    const int bf16 = a.ab_bf16;
    int blk = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const int nk = a.items[it].w;
      for (int j = 0; j < nk; ++j, ++blk) {
        const int st = blk % ns, us = blk / ns;
        // the four warps agree on the outcome, so that all 128 threads or
        // none reach the NVFP4 barrier below
        ok = widen_all(mbar_wait(&c.stg_full[st], us & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        const int valid = c.info[st].valid;
        const uint32_t kst = sbase + st * kStage, vst = kst + kKVTile;
        if (kKV == kKvFp4) {
          if (k < valid) {
            widen_fp4_row(vst + k * 64, vst + 8192 + k * 8, kst, k, bf16);
          } else {
            for (int ch = 0; ch < 16; ++ch) st_shared_v4(kst + swz_kv(k, ch), 0, 0, 0, 0);
          }
          uint4 vc[4];
          uint2 vs = make_uint2(0u, 0u);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c4 = (cc + k) & 3;  // rotated to spread banks
            vc[cc] = k < valid ? ld_shared_v4(vst + 16384 + k * 64 + c4 * 16) : make_uint4(0, 0, 0, 0);
          }
          if (k < valid) vs = ld_shared_v2(vst + 16384 + 8192 + k * 8);
          widen_sync();  // every V row read before any is written
          if (k < valid) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) widen_fp4_chunk(vc[cc], vs, vst, k, (cc + k) & 3, bf16);
          } else {
            for (int ch = 0; ch < 16; ++ch) st_shared_v4(vst + swz_kv(k, ch), 0, 0, 0, 0);
          }
        } else {
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t src = vst + kv * 16384 + k * 128;
            const uint32_t dst = kv ? vst : kst;
            uint4 raw[8];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)  // rotated to spread banks
              raw[cc] = k < valid ? ld_shared_v4(src + ((cc + k) & 7) * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              const int c8 = (cc + k) & 7;
              const uint32_t w[4] = {raw[cc].x, raw[cc].y, raw[cc].z, raw[cc].w};
              uint32_t o[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                o[2 * i] = widen_e4m3x2((uint16_t)(w[i] & 0xffffu), bf16);
                o[2 * i + 1] = widen_e4m3x2((uint16_t)(w[i] >> 16), bf16);
              }
              st_shared_v4(dst + swz_kv(k, 2 * c8), o[0], o[1], o[2], o[3]);
              st_shared_v4(dst + swz_kv(k, 2 * c8 + 1), o[4], o[5], o[6], o[7]);
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&c.kv_full[st]);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------ softmax group
    // Each thread waits on the barriers itself; the four warps vote once per
    // block (an abort, or a score above the running maximum anywhere), so
    // every named barrier below is reached by all 128 threads or by none.
    const int k = tid;  // key of S^T / head dim of O^T / TMEM lane
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const int bf16 = a.ab_bf16;
    const float c2 = a.scale_log2;
    const int G = a.G;
    const uint32_t kk = (uint32_t)(k & 63);
    // byte offset of key k in row r of a [rows][keys] P^T tile: 128-byte
    // swizzled K-major, two halves of 64 keys
    const uint32_t p_key = (uint32_t)(k >> 6) * (uint32_t)(N * 128) + (kk & 7u) * 2u;
    int blk = 0, n_it = 0;
    bool ok = true;
    float m[N], lsum[N];
    // The epilogue of an item (o = O / l into its partial rows) waits for
    // the item's last p v, so it runs at the end of the next item (the O
    // accumulators alternate between items; the next-but-one item's first
    // p v needs it, and comes after it); the CTA's last item finishes at
    // once.  An item's sums wait in shared memory, ordered by the named
    // barriers in between.
    static_assert(N <= 16, "inv_l holds 16 rows");
    int prev_e0 = 0;
    auto finish = [&](int pn, int pend_e0) -> bool {
      const int pend_ib = pn & 1, pend_ui = pn >> 1;
      const uint32_t tOp = tmem + lane_addr + 2 * N + pend_ib * N;
      const bool oko = __all_sync(
          0xffffffffu, mbar_wait(&c.o_full[pend_ib], pend_ui & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
      float o[N];
      if (oko) {
        tc_fence_after();
        tmem_ld_n<N>(tOp, o);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&c.o_empty[pend_ib]);
      }
      if (!wg_all(oko)) return false;
      // o = O / l (thread k: head dim k of every row), FP32 or rounded to
      // the q dtype
      const size_t o0 = (size_t)pend_e0 * G * 128 + k;
#pragma unroll
      for (int r = 0; r < N; ++r) {
        if (r >= G) continue;
        const float ov = o[r] * c.inv_l[pend_ib][r];
        if (kPart32) {
          __stcs(static_cast<float*>(a.part_o) + o0 + (size_t)r * 128, ov);
        } else {
          const unsigned short h =
              bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(ov)) : __half_as_ushort(__float2half_rn(ov));
          __stcs(static_cast<unsigned short*>(a.part_o) + o0 + (size_t)r * 128, h);
        }
      }
      if (k < G) a.part_lse[(size_t)pend_e0 * G + k] = c.lse[pend_ib][k];
      return true;
    };
    int4 itm_next = a.items[it_begin];
    for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
      const int4 itm = itm_next;
      if (it + 1 < it_end) itm_next = a.items[it + 1];  // its latency hides behind this item
      const int nk = itm.w;
      const int ib = n_it & 1;
      const uint32_t tO = tmem + lane_addr + 2 * N + ib * N;
      for (int j = 0; j < nk; ++j, ++blk) {
        const int st = blk % ns, us = blk / ns, sb = blk & 1, ub = blk >> 1;
        uint8_t* kst = sm + st * kStage;
        uint8_t* vst = kst + kKVTile;
        int valid = 0;
        bool okb;
        // the block's K and V in stage st (widened caches: written by the
        // widening warps, which zero the rows past the valid keys)
        okb = mbar_wait(&c.kv_full[st], us & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        if (okb) {
          valid = c.info[st].valid;
          if (kKV == kKv16 && k >= valid) {
            // keys past the sequence end must not bring stale values into P V
            for (int ch = 0; ch < 16; ++ch) st_shared_v4(smem_u32(vst) + swz_kv(k, ch), 0, 0, 0, 0);
          }
        }
        // ---- scores of key k for every row (tcgen05.ld is warp-collective)
        okb = __all_sync(0xffffffffu,
                         okb && mbar_wait(&c.s_full[sb], ub & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        float x[N];
        if (okb) {
          tc_fence_after();
          tmem_ld_n<N>(tmem + lane_addr + sb * N, x);
          tmem_ld_wait();
        }
#pragma unroll
        for (int r = 0; r < N; ++r) x[r] = (okb && k < valid && r < G) ? x[r] * c2 : -INFINITY;
        bool exceed = false;
        if (j > 0) {
#pragma unroll
          for (int r = 0; r < N; ++r) exceed |= x[r] > m[r] + kRescaleThreshold;
        }
        okb = okb && mbar_wait(&c.p_empty[sb], (ub & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        if (j == 0 || wg_any(exceed || !okb)) {
          if (!wg_all(okb)) {
            ok = false;
            break;
          }
          if (j == 0) {
#pragma unroll
            for (int r = 0; r < N; ++r) m[r] = x[r];
            wg_reduce<N, true>(m, red);
#pragma unroll
            for (int r = 0; r < N; ++r) {
              if (m[r] == -INFINITY) m[r] = 0.f;  // padding rows
              lsum[r] = 0.f;
            }
          } else {
            // raise m: wait until the previous P V finished, rescale O^T
            float mb[N];
#pragma unroll
            for (int r = 0; r < N; ++r) mb[r] = x[r];
            wg_reduce<N, true>(mb, red);
            const int pb = blk - 1;
            ok = wg_all(mbar_wait(&c.p_empty[pb & 1], (pb >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT,
                                  kWaitLimitNs));
            if (!ok) break;
            tc_fence_after();
            float alpha[N], o[N];
#pragma unroll
            for (int r = 0; r < N; ++r) {
              const float mn = fmaxf(m[r], mb[r]);
              alpha[r] = ex2_approx(m[r] - mn);
              m[r] = mn;
              lsum[r] *= alpha[r];
            }
            tmem_ld_n<N>(tO, o);
            tmem_ld_wait();
#pragma unroll
            for (int r = 0; r < N; ++r) o[r] *= alpha[r];
            tmem_st_n<N>(tO, o);
          }
        }
        // ---- P^T of key k into the [rows][keys] operand tile
        const uint32_t pbuf = smem_u32(sm + L.p + sb * (N * 256)) + p_key;
#pragma unroll
        for (int r = 0; r < N; ++r) {
          const float pr = x[r] == -INFINITY ? 0.f : ex2_approx(x[r] - m[r]);
          lsum[r] += pr;
          const uint16_t h = bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(pr)) : __half_as_ushort(__float2half_rn(pr));
          st_shared_u16(pbuf + (uint32_t)r * 128u + (((kk >> 3) ^ (uint32_t)(r & 7)) << 4), h);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&c.p_full[sb]);
      }
      if (!ok) break;
      // ---- the item's sums: l over the four warps, 1 / l per row and
      // lse = (m + log2 l) ln 2; its epilogue follows the next item's first
      // softmax, or now for the last item
      wg_reduce<N, false>(lsum, red);
      if (k == 0) {  // every thread holds the same sums; read after the next named barrier
#pragma unroll
        for (int r = 0; r < N; ++r) c.inv_l[ib][r] = lsum[r] > 0.f ? __frcp_rn(lsum[r]) : 0.f;
      }
      if (k < G) {
        float lv = -INFINITY, mv = 0.f;
#pragma unroll
        for (int r = 0; r < N; ++r)
          if (r == k) {
            lv = lsum[r];
            mv = m[r];
          }
        c.lse[ib][k] = lv > 0.f ? (mv + lg2_approx(lv)) * 0.69314718055994530942f : -INFINITY;
      }
      // the previous item's epilogue (its last p v finished long ago), and
      // this one's when it is the CTA's last item
      for (int q = n_it > 0 ? n_it - 1 : 0; q <= (it + 1 == it_end ? n_it : n_it - 1) && ok; ++q)
        ok = finish(q, q == n_it ? itm.y : prev_e0);
      prev_e0 = itm.y;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {  // every barrier this phase initialised
    for (int i = 0; i < ns; ++i) {
      mbar_inval(&c.kv_full[i]);
      mbar_inval(&c.kv_empty[i]);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_inval(&c.q_full[i]);
      mbar_inval(&c.q_empty[i]);
      mbar_inval(&c.s_full[i]);
      mbar_inval(&c.p_full[i]);
      mbar_inval(&c.p_empty[i]);
      mbar_inval(&c.o_full[i]);
      mbar_inval(&c.o_empty[i]);
    }
    for (int i = 0; i < ns; ++i) mbar_inval(&c.stg_full[i]);
    mbar_inval(&c.done);
  }
  __syncthreads();
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

inline bool make_q_map(CUtensorMap* m, const void* q, const mxsa_problem& p, int n_rows_box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)p.total_q * p.num_q_heads};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, (cuuint32_t)n_rows_box};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapDataType dt = p.q_dtype == MXSA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, dt, 2, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Smallest dynamic shared memory (plus 1024 for alignment) the decode
// phase needs for the cache dtype.
inline size_t smem_bytes(bool fp8) {
  constexpr int N = 16;
  return smem_layout<N>(stages_for<N>(fp8 ? 1 : 0)).total + 1024;
}

// Fills the decode phase's arguments and its q tensor map; false when the
// tensor map cannot be made.
inline bool make_args(const mxsa_problem& p, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const IndexPtrs& ix, const SchedPtrs& sc, void* part_o,
                      float* part_lse, DecArgs* a, CUtensorMap* tmq) {
  constexpr int N = 16;
  const int G = p.num_q_heads / p.num_kv_heads;
  *a = DecArgs{};
  std::memset(tmq, 0, sizeof(*tmq));
  if (G > kDecodeMaxG || p.total_q == 0) return true;  // no decode item can exist: phase off (cta_ptr null)
  if (!make_q_map(tmq, q, p, N)) return false;
  a->block_tables = block_tables;
  a->seq = ix.seq;
  a->active = ix.active;
  a->row_ptr = ix.row_ptr;
  a->items = sc.items_dec;
  a->cta_ptr = sc.cta_ptr_dec;
  a->idx_hdr = ix.hdr;
  a->sch_hdr = sc.hdr;
  a->part_o = part_o;
  a->part_lse = part_lse;
  a->flags = ix.hdr + kHdrFlags;
  a->num_seqs = p.num_seqs;
  a->Hq = p.num_q_heads;
  a->Hkv = p.num_kv_heads;
  a->G = G;
  a->page_size = p.page_size;
  a->max_pages = p.max_pages_per_seq;
  a->num_pages = p.num_pages;
  a->kv_fp8 = kv_widened(p) ? 1 : 0;
  a->kv_fp4 = p.kv_dtype == MXSA_NVFP4 ? 1 : 0;
  a->kbase = static_cast<const uint8_t*>(k_cache);
  a->vbase = static_cast<const uint8_t*>(v_cache);
  a->ab_bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
  a->ns = stages_for<N>(a->kv_fp8);
  a->part32 = partials_fp32(p) ? 1 : 0;
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 0.08838834764831845f;  // 1/sqrt(128)
  a->scale_log2 = scale * 1.4426950408889634f;
  return true;
}

}  // namespace dec

}  // namespace mxsa
