// KV-outer forward (fw-ai/minimax-kernels README, intro: "loads a selected
// KV block once and processes all queries that selected it").
//
// Persistent kernel, one CTA per SM, 192 threads:
//   warps 0-3  softmax warpgroup: gathers the q rows of a tile into shared
//              memory, turns S = q k^T (TMEM) into P = exp(S - m) (shared
//              memory), and writes o = (P v) / l and lse per row; for FP8
//              caches it also widens the staged e4m3 block to BF16/FP16.
//   warp 4     TMA producer: decodes the work item (key -> kv head,
//              sequence, block), walks the block table and loads the 1-2
//              pages of K and V of the block into a double-buffered stage.
//   warp 5     TMEM owner and MMA issuer (tcgen05.mma, cta_group::1,
//              M = N = 128, K = 16 per instruction, FP32 accumulate):
//              S = Q K^T into TMEM columns [0,128), O = P V into [128,256).
//
// Rows of a tile are (entry, head) pairs: up to 128 / G consecutive entries
// of the item's key, each contributing its G query heads.  Row r of the
// tile is TMEM lane r and is owned by softmax thread r.
//
// Shared-memory operands use the 128-byte swizzled K-major layout (q, K, P)
// and the 128-byte swizzled MN-major layout (V as the B operand of P V).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mxsa {

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = 32768;  // 128 rows x 128 x 16-bit
constexpr uint32_t kStageBytes = 2 * kTileBytes;

struct ItemInfo {
  int32_t g, s, b, valid, e0, n, L, tq, q_begin, absent, pad0, pad1, pad2, pad3, pad4, pad5;
};

struct Ctrl {
  uint64_t kv_full[2], kv_empty[2], stg_full, stg_empty, q_full, s_full, p_full, o_full, done;
  uint32_t tmem_base;
  int32_t abort_flag;
  ItemInfo info[2];
};

struct FwdArgs {
  const uint8_t* q;
  const int32_t* block_tables;
  const SeqInfo* seq;
  const int32_t* entries;
  const int4* items;
  const int32_t* cta_ptr;
  const int32_t* idx_hdr;
  const int32_t* sch_hdr;
  float* part_o;
  float* part_lse;
  int32_t* flags;
  int32_t num_seqs, Hq, Hkv, G, topk, page_size, max_pages, num_pages, causal, kv_fp8, ab_bf16, per_tile;
  float scale_log2;
};

// smem offsets from the 1024-aligned base
constexpr uint32_t kOffKV = 0;                             // 2 stages x (K, V)
constexpr uint32_t kOffQ = 2 * kStageBytes;                // 131072
constexpr uint32_t kOffP = kOffQ + kTileBytes;             // 163840
constexpr uint32_t kOffStg = kOffP + kTileBytes;           // 196608 (FP8 staging, 32 KB)
constexpr uint32_t kCtrlBf16 = kOffStg;                    // control block without staging
constexpr uint32_t kCtrlFp8 = kOffStg + kTileBytes;        // 229376

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

__global__ void __launch_bounds__(kThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl& c = *reinterpret_cast<Ctrl*>(sm + (a.kv_fp8 ? kCtrlFp8 : kCtrlBf16));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  pdl_wait();  // the schedule (and the previous forward) are complete

  if (a.sch_hdr[kSchCtas] != (int)gridDim.x) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(a.flags, MXSA_FLAG_SCHEDULE);
    return;
  }
  const int it_begin = a.cta_ptr[blockIdx.x], it_end = a.cta_ptr[blockIdx.x + 1];
  if (it_begin >= it_end) return;  // uniform: nothing to do, nothing allocated

  if (tid == 0) {
    mbar_init(&c.kv_full[0], a.kv_fp8 ? 128 : 1);
    mbar_init(&c.kv_full[1], a.kv_fp8 ? 128 : 1);
    mbar_init(&c.kv_empty[0], 1);
    mbar_init(&c.kv_empty[1], 1);
    mbar_init(&c.stg_full, 1);
    mbar_init(&c.stg_empty, 128);
    mbar_init(&c.q_full, 128);
    mbar_init(&c.s_full, 1);
    mbar_init(&c.p_full, 128);
    mbar_init(&c.o_full, 1);
    mbar_init(&c.done, 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&c.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  volatile int* abort_flag = &c.abort_flag;
  const uint32_t sbase = smem_u32(sm);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const int NB = a.idx_hdr[kHdrNB];
      const int ps = a.page_size;
      int n = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++n) {
        const int st = n & 1, use = n >> 1;
        ok = mbar_wait(&c.kv_empty[st], (use & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        if (!ok) break;
        const int4 itm = a.items[it];
        const int key = itm.x;
        const int g = key / NB, r = key - g * NB;
        const int s = seq_of_block(a.seq, a.num_seqs, r);
        const SeqInfo si = a.seq[s];
        const int b = r - si.blk_off;
        const int valid = min(128, si.L - 128 * b);
        // physical pages of the block (1 for 128-token pages, 1-2 for 64)
        int pages[2] = {-1, -1};
        int absent = 0;
        const int npg = ps == 128 ? 1 : 2;
        for (int pg = 0; pg < npg; ++pg) {
          const bool needed = pg * 64 < valid;
          if (!needed) {
            absent |= 1 << pg;
            continue;
          }
          const int lp = ps == 128 ? b : 2 * b + pg;
          const int phys = a.block_tables[(size_t)s * a.max_pages + lp];
          if (phys < 0 || phys >= a.num_pages) {
            atomicOr(a.flags, MXSA_FLAG_PAGE);
            absent |= 1 << pg;
            continue;
          }
          pages[pg] = phys;
        }
        ItemInfo inf;
        inf.g = g; inf.s = s; inf.b = b; inf.valid = valid; inf.e0 = itm.y; inf.n = itm.z;
        inf.L = si.L; inf.tq = si.tq; inf.q_begin = si.q_begin; inf.absent = absent;
        c.info[st] = inf;
        const int present = (pages[0] >= 0) + (pages[1] >= 0);
        if (!a.kv_fp8) {
          const uint32_t bytes = (uint32_t)present * (uint32_t)ps * 512u;  // K+V, both halves
          uint8_t* kdst = sm + kOffKV + st * kStageBytes;
          uint8_t* vdst = kdst + kTileBytes;
          mbar_arrive_expect_tx(&c.kv_full[st], bytes);
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            const int z = pages[pg] * a.Hkv + g;
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(kdst + h * 16384 + pg * 8192, &tmk, &c.kv_full[st], h * 64, 0, z);
              tma_load_3d(vdst + h * 16384 + pg * 8192, &tmv, &c.kv_full[st], h * 64, 0, z);
            }
          }
        } else {
          ok = mbar_wait(&c.stg_empty, (n & 1) ^ 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (!ok) break;
          const uint32_t bytes = (uint32_t)present * (uint32_t)ps * 256u;
          uint8_t* stg = sm + kOffStg;
          mbar_arrive_expect_tx(&c.stg_full, bytes);
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            const int z = pages[pg] * a.Hkv + g;
            tma_load_3d(stg + pg * 8192, &tmk, &c.stg_full, 0, 0, z);
            tma_load_3d(stg + 16384 + pg * 8192, &tmv, &c.stg_full, 0, 0, z);
          }
        }
      }
      // drain: wait until every load this thread issued has landed
      for (int k = std::max(0, n - 2); k < n; ++k) {
        if (a.kv_fp8) {
          if (k == n - 1) mbar_wait(&c.stg_full, k & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        } else {
          mbar_wait(&c.kv_full[k & 1], (k >> 1) & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        }
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16(128, 128, (uint32_t)a.ab_bf16, 0, 0);
      const uint32_t id_pv = idesc_f16(128, 128, (uint32_t)a.ab_bf16, 0, 1);
      const uint32_t tS = tmem, tO = tmem + 128;
      const uint32_t q_s = sbase + kOffQ, p_s = sbase + kOffP;
      int n = 0;
      uint32_t tile_ctr = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++n) {
        const int st = n & 1, use = n >> 1;
        ok = mbar_wait(&c.kv_full[st], use & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        const int n_entries = c.info[st].n;
        const int ntiles = (n_entries + a.per_tile - 1) / a.per_tile;
        const uint32_t k_s = sbase + kOffKV + st * kStageBytes, v_s = k_s + kTileBytes;
        for (int j = 0; j < ntiles; ++j, ++tile_ctr) {
          ok = mbar_wait(&c.q_full, tile_ctr & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
            mma_f16_ss(tS, smem_desc_sw128(q_s + off, 0, 1024), smem_desc_sw128(k_s + off, 0, 1024), id_qk,
                       ks > 0);
          }
          mma_commit(&c.s_full);
          ok = mbar_wait(&c.p_full, tile_ctr & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
            mma_f16_ss(tO, smem_desc_sw128(p_s + off, 0, 1024),
                       smem_desc_sw128(v_s + ks * 2048u, 16384, 1024), id_pv, ks > 0);
          }
          mma_commit(&c.o_full);
        }
        mma_commit(&c.kv_empty[st]);
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      mma_commit(&c.done);
      mbar_wait(&c.done, 0, abort_flag, a.flags, MXSA_FLAG_TIMEOUT, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------ softmax group
    const int r = tid;  // tile row == TMEM lane
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const int bf16 = a.ab_bf16;
    int n = 0;
    uint32_t tile_ctr = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n) {
      const int st = n & 1, use = n >> 1;
      uint8_t* kst = sm + kOffKV + st * kStageBytes;
      uint8_t* vst = kst + kTileBytes;
      ItemInfo inf;
      if (a.kv_fp8) {
        ok = __all_sync(0xffffffffu, mbar_wait(&c.stg_full, n & 1, abort_flag, a.flags, MXSA_FLAG_TIMEOUT,
                                                kWaitLimitNs));
        if (!ok) break;
        inf = c.info[st];
        // widen row r of the staged K and V (e4m3, 128 B per row) into the
        // swizzled 16-bit operand tiles; rows past the valid tokens become 0
        const uint8_t* stg = sm + kOffStg;
        for (int kv = 0; kv < 2; ++kv) {
          const uint8_t* src = stg + kv * 16384 + r * 128;
          uint8_t* dst = kv ? vst : kst;
          for (int cc = 0; cc < 8; ++cc) {
            const int c8 = (cc + r) & 7;  // rotate to spread banks
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (r < inf.valid) raw = *reinterpret_cast<const uint4*>(src + c8 * 16);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[2 * i] = widen_e4m3x2((uint16_t)(w[i] & 0xffffu), bf16);
              o[2 * i + 1] = widen_e4m3x2((uint16_t)(w[i] >> 16), bf16);
            }
            // 16 fp8 -> 16 x 16-bit = chunks 2*c8 and 2*c8+1 of the row
            st_shared_v4(smem_u32(dst) + swz(r, 2 * c8), o[0], o[1], o[2], o[3]);
            st_shared_v4(smem_u32(dst) + swz(r, 2 * c8 + 1), o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&c.stg_empty);
        mbar_arrive(&c.kv_full[st]);
      } else {
        ok = __all_sync(0xffffffffu, mbar_wait(&c.kv_full[st], use & 1, abort_flag, a.flags,
                                                MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        inf = c.info[st];
        if (r >= inf.valid) {
          // keys past the sequence end (or of a skipped page) must not carry
          // stale values into P V: zero row r of V
          for (int ch = 0; ch < 16; ++ch) st_shared_v4(smem_u32(vst) + swz(r, ch), 0, 0, 0, 0);
        }
      }
      const int ntiles = (inf.n + a.per_tile - 1) / a.per_tile;
      for (int j = 0; j < ntiles; ++j, ++tile_ctr) {
        const int et0 = inf.e0 + j * a.per_tile;
        const int ne = min(a.per_tile, inf.n - j * a.per_tile);
        const int rows = ne * a.G;
        // ---- gather q rows into the swizzled Q tile
        int lim = 0;
        size_t orow = 0;
        if (r < rows) {
          const int e = et0 + r / a.G, hh = r % a.G;
          const int slot = a.entries[e];
          const int t = slot / (a.Hkv * a.topk);
          const int h = inf.g * a.G + hh;
          const uint4* src = reinterpret_cast<const uint4*>(a.q + ((size_t)t * a.Hq + h) * 256);
          uint4 v[16];
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) v[ch] = __ldg(src + ch);
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) st_shared_v4(sbase + kOffQ + swz(r, ch), v[ch].x, v[ch].y, v[ch].z, v[ch].w);
          const int pos = inf.L - inf.tq + (t - inf.q_begin);
          lim = inf.valid;
          if (a.causal) lim = min(lim, pos - 128 * inf.b + 1);
          orow = (size_t)e * a.G + hh;
        } else {
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) st_shared_v4(sbase + kOffQ + swz(r, ch), 0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        mbar_arrive(&c.q_full);
        // ---- softmax of the row
        ok = __all_sync(0xffffffffu, mbar_wait(&c.s_full, tile_ctr & 1, abort_flag, a.flags,
                                                MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        float m2 = -INFINITY, l = 0.f;
        if (warp * 32 < rows) {
          float sv[128];
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tmem_ld32(tmem + lane_addr + cb * 32, sv + cb * 32);
          tmem_ld_wait();
          if (r < rows) {
            float m = -INFINITY;
#pragma unroll
            for (int k = 0; k < 128; ++k)
              if (k < lim) m = fmaxf(m, sv[k]);
            m2 = m * a.scale_log2;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
              uint32_t pk[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int k0 = ch * 8 + 2 * i;
                const float p0 = k0 < lim ? ex2_approx(fmaf(sv[k0], a.scale_log2, -m2)) : 0.f;
                const float p1 = k0 + 1 < lim ? ex2_approx(fmaf(sv[k0 + 1], a.scale_log2, -m2)) : 0.f;
                l += p0 + p1;
                pk[i] = pack2(p0, p1, bf16);
              }
              st_shared_v4(sbase + kOffP + swz(r, ch), pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
        if (r >= rows) {
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) st_shared_v4(sbase + kOffP + swz(r, ch), 0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&c.p_full);
        // ---- epilogue: o = O / l, lse = (m2 + log2 l) * ln 2
        ok = __all_sync(0xffffffffu, mbar_wait(&c.o_full, tile_ctr & 1, abort_flag, a.flags,
                                                MXSA_FLAG_TIMEOUT, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        if (warp * 32 < rows) {
          // every indexed row has at least one key; l == 0 only on corrupt input
          const float inv_l = l > 0.f ? 1.f / l : 0.f;
          float4* dst = reinterpret_cast<float4*>(a.part_o + orow * 128);
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) {
            float ov[32];
            tmem_ld32(tmem + lane_addr + 128 + cb * 32, ov);
            tmem_ld_wait();
            if (r < rows) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[cb * 8 + i] = make_float4(ov[4 * i] * inv_l, ov[4 * i + 1] * inv_l, ov[4 * i + 2] * inv_l,
                                              ov[4 * i + 3] * inv_l);
            }
          }
          if (r < rows) a.part_lse[orow] = l > 0.f ? (m2 + lg2_approx(l)) * 0.69314718055994530942f : -INFINITY;
        }
        tc_fence_before();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 3-D view of a cache [pages * Hkv][page_size][128]: box = one page, one
// 128-byte column slab (64 x 16-bit, swizzled) or the full 128 e4m3 row.
bool make_cache_map(CUtensorMap* m, const void* base, const mxsa_problem& p) {
  auto fn = encode_fn();
  if (!fn) return false;
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

size_t fwd_smem_bytes(bool fp8) { return (fp8 ? kCtrlFp8 : kCtrlBf16) + sizeof(Ctrl) + 1024; }

cudaError_t launch_fwd(const mxsa_problem& p, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const IndexPtrs& ix, const SchedPtrs& sc, int num_ctas,
                       float* part_o, float* part_lse, cudaStream_t st, int* err_detail) {
  CUtensorMap tmk, tmv;
  if (!make_cache_map(&tmk, k_cache, p) || !make_cache_map(&tmv, v_cache, p)) {
    *err_detail = 1;
    return cudaErrorInvalidValue;
  }
  // decode work items (runs of single-token keys) first, then the
  // KV-stationary items; each kernel's CTAs without items exit at once
  cudaError_t de = launch_fwd_decode(p, q, tmk, tmv, block_tables, ix, sc, num_ctas, part_o, part_lse, st,
                                     err_detail);
  if (de != cudaSuccess) return de;
  const bool fp8 = p.kv_dtype == MXSA_FP8_E4M3;
  const size_t smem = fwd_smem_bytes(fp8);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)fwd_smem_bytes(true));
  });
  if (attr_err != cudaSuccess) return attr_err;
  FwdArgs a;
  a.q = static_cast<const uint8_t*>(q);
  a.block_tables = block_tables;
  a.seq = ix.seq;
  a.entries = ix.entries;
  a.items = sc.items;
  a.cta_ptr = sc.cta_ptr;
  a.idx_hdr = ix.hdr;
  a.sch_hdr = sc.hdr;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.flags = ix.hdr + kHdrFlags;
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
  a.ab_bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
  a.per_tile = std::max(1, MXSA_TILE_ROWS / a.G);
  const float scale = p.softmax_scale > 0.f ? p.softmax_scale : 0.08838834764831845f;  // 1/sqrt(128)
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_pdl(k_fwd, dim3(num_ctas), dim3(kThreads), smem, st, tmk, tmv, a);
}

}  // namespace mxsa
