// Combine: LSE-weighted merge of the per-block partials of every (token,
// head) row ("combine" kernel in the test list of the fw-ai/minimax-kernels
// README; output [Tq, Hq, 128] and FP32 lse [Hq, Tq] from its Quick start).
//
//   M = max_k lse_k,  w_k = exp(lse_k - M),
//   out = sum_k w_k o_k / sum_k w_k   (rounded to nearest-even, q dtype),
//   lse = M + log(sum_k w_k);  no partial: out = 0, lse = -inf.
//
// Partial rows hold 128 FP32 values, or 128 values of the 16-bit q dtype
// (widened exactly to FP32 here), and an FP32 lse.  One warp per row; lane
// j owns columns 4j..4j+3 (16 or 8 bytes of every partial row, so each
// partial is read as one coalesced transaction of the whole row, up to 8 of
// them in flight per warp).  The row's slot -> entry map and lses are read
// once per 32 slots with one load per lane.  With top-k <= 32 a second form
// (k_combine_small) keeps each warp one row ahead on those reads, so only
// the partial rows' own reads sit in a row's path.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace mxsa {

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kBatch = 8;  // partial rows read ahead per warp

// four 16-bit values (bf16 or fp16, low half first) -> FP32, exactly
__device__ __forceinline__ float4 widen4(uint2 raw, int bf16) {
  if (bf16)
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// one lane's four columns of a partial row
template <typename P>
struct PartialCols;
template <>
struct PartialCols<float> {
  using raw_t = float4;
  static __device__ __forceinline__ raw_t zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  static __device__ __forceinline__ float4 widen(raw_t v, int) { return v; }
};
template <>
struct PartialCols<uint16_t> {
  using raw_t = uint2;
  static __device__ __forceinline__ raw_t zero() { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ float4 widen(raw_t v, int bf16) { return widen4(v, bf16); }
};

template <typename P>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 4)
    k_combine(const int32_t* slot_entry, const P* part_o, const float* part_lse, uint8_t* out, float* lse_out,
              int total_q, int Hq, int Hkv, int topk, int out_bf16) {
  using PC = PartialCols<P>;
  const int lane = threadIdx.x & 31;
  const int G = Hq / Hkv;
  const long long n_rows = (long long)total_q * Hq;
  pdl_wait();  // the forward's partials are complete
  constexpr float kLog2e = 1.4426950408889634f;
  for (long long row = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); row < n_rows;
       row += (long long)gridDim.x * kWarpsPerBlock) {
    const int t = (int)(row / Hq), h = (int)(row % Hq);
    const int g = h / G, j = h % G;
    const int32_t* se = slot_entry + ((long long)t * Hkv + g) * topk;
    // pass 1: max lse over the row's partials
    float M = -INFINITY;
    for (int k0 = 0; k0 < topk; k0 += 32) {
      const int k = k0 + lane;
      float l = -INFINITY;
      if (k < topk) {
        const int e = se[k];
        if (e >= 0) l = part_lse[(long long)e * G + j];
      }
      M = fmaxf(M, l);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    if (M != -INFINITY) {
      const float M2 = M * kLog2e;
      for (int k0 = 0; k0 < topk; k0 += 32) {
        const int k = k0 + lane;
        int e = -1;
        float w = 0.f;
        if (k < topk) {
          e = se[k];
          if (e >= 0) {
            const float l = part_lse[(long long)e * G + j];
            w = l == -INFINITY ? 0.f : ex2_approx(fmaf(l, kLog2e, -M2));
          }
        }
        unsigned live = __ballot_sync(0xffffffffu, w > 0.f);
        while (live) {
          // up to kBatch partial rows are requested before any is used, so
          // that each warp keeps several whole-row reads in flight; they are
          // accumulated in slot order (absent ones add exact zeros)
          typename PC::raw_t v[kBatch];
          float ws[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            ws[u] = 0.f;
            v[u] = PC::zero();
            if (live) {  // warp-uniform
              const int src = __ffs(live) - 1;
              live &= live - 1;
              const int es = __shfl_sync(0xffffffffu, e, src);
              ws[u] = __shfl_sync(0xffffffffu, w, src);
              v[u] = __ldcs(reinterpret_cast<const typename PC::raw_t*>(part_o + ((long long)es * G + j) * 128) + lane);
            }
          }
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const float4 f = PC::widen(v[u], out_bf16);
            acc.x = fmaf(ws[u], f.x, acc.x);
            acc.y = fmaf(ws[u], f.y, acc.y);
            acc.z = fmaf(ws[u], f.z, acc.z);
            acc.w = fmaf(ws[u], f.w, acc.w);
            W += ws[u];
          }
        }
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint2 packed;
    if (out_bf16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      packed = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    } else {
      __half2 a = __floats2half2_rn(acc.x * inv, acc.y * inv);
      __half2 b = __floats2half2_rn(acc.z * inv, acc.w * inv);
      packed = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
    reinterpret_cast<uint2*>(out + row * 256)[lane] = packed;
    if (lse_out && lane == 0)
      lse_out[(long long)h * total_q + t] = W > 0.f ? M + lg2_approx(W) * 0.69314718055994530942f : -INFINITY;
  }
}

// The same merge when every row has at most 32 slots (top-k <= 32): lane k
// holds slot k's entry and lse, and each warp works one row ahead, so a
// row's slot -> entry map and lses are in registers when its partial rows
// are requested.  The next row's map is requested before this row's
// partials, its lses once the map has landed (after this row's first
// batch); the partials themselves are read and summed exactly as above.
// 16-bit rows are half as large: 12 of them are requested per batch, which
// still fits four CTAs per SM (measured on a 32-partial prefill against 8
// per batch, and against 16 or 20 at three CTAs per SM, which lose more to
// the lower occupancy than the deeper batch gains).
template <typename P>
constexpr int small_batch() { return sizeof(P) == 2 ? 12 : kBatch; }

template <typename P>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 4)
    k_combine_small(const int32_t* slot_entry, const P* part_o, const float* part_lse, uint8_t* out,
                    float* lse_out, int total_q, int Hq, int Hkv, int topk, int out_bf16) {
  using PC = PartialCols<P>;
  const int lane = threadIdx.x & 31;
  const int G = Hq / Hkv;
  const long long n_rows = (long long)total_q * Hq;
  const long long stride = (long long)gridDim.x * kWarpsPerBlock;
  constexpr float kLog2e = 1.4426950408889634f;
  // slot `lane` of row `row`: its entry (-1: none)
  auto entry_of = [&](long long row) -> int {
    if (row >= n_rows || lane >= topk) return -1;
    const int t = (int)(row / Hq), h = (int)(row % Hq);
    return slot_entry[((long long)t * Hkv + h / G) * topk + lane];
  };
  auto lse_of = [&](long long row, int e) -> float {
    return e >= 0 ? part_lse[(long long)e * G + (int)(row % Hq) % G] : -INFINITY;
  };
  pdl_wait();  // the forward's partials are complete
  long long row = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  int e_next = entry_of(row);
  float l_next = lse_of(row, e_next);
  for (; row < n_rows; row += stride) {
    const int t = (int)(row / Hq), h = (int)(row % Hq);
    const int j = h % G;
    const int e = e_next;
    const float l = l_next;
    const long long nrow = row + stride;
    e_next = entry_of(nrow);
    float M = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    bool next_lse = false;
    if (M != -INFINITY) {
      const float M2 = M * kLog2e;
      const float w = (e >= 0 && l != -INFINITY) ? ex2_approx(fmaf(l, kLog2e, -M2)) : 0.f;
      unsigned live = __ballot_sync(0xffffffffu, w > 0.f);
      while (live) {
        typename PC::raw_t v[small_batch<P>()];
        float ws[small_batch<P>()];
#pragma unroll
        for (int u = 0; u < small_batch<P>(); ++u) {
          ws[u] = 0.f;
          v[u] = PC::zero();
          if (live) {  // warp-uniform
            const int src = __ffs(live) - 1;
            live &= live - 1;
            const int es = __shfl_sync(0xffffffffu, e, src);
            ws[u] = __shfl_sync(0xffffffffu, w, src);
            v[u] = __ldcs(reinterpret_cast<const typename PC::raw_t*>(part_o + ((long long)es * G + j) * 128) + lane);
          }
        }
#pragma unroll
        for (int u = 0; u < small_batch<P>(); ++u) {
          const float4 f = PC::widen(v[u], out_bf16);
          acc.x = fmaf(ws[u], f.x, acc.x);
          acc.y = fmaf(ws[u], f.y, acc.y);
          acc.z = fmaf(ws[u], f.z, acc.z);
          acc.w = fmaf(ws[u], f.w, acc.w);
          W += ws[u];
        }
        if (!next_lse) {
          l_next = lse_of(nrow, e_next);
          next_lse = true;
        }
      }
    }
    if (!next_lse) l_next = lse_of(nrow, e_next);
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint2 packed;
    if (out_bf16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 b = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      packed = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    } else {
      __half2 a = __floats2half2_rn(acc.x * inv, acc.y * inv);
      __half2 b = __floats2half2_rn(acc.z * inv, acc.w * inv);
      packed = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
    reinterpret_cast<uint2*>(out + row * 256)[lane] = packed;
    if (lse_out && lane == 0)
      lse_out[(long long)h * total_q + t] = W > 0.f ? M + lg2_approx(W) * 0.69314718055994530942f : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_combine(const mxsa_problem& p, const IndexPtrs& ix, const void* part_o,
                           const float* part_lse, void* out, float* lse, cudaStream_t st) {
  const long long rows = (long long)p.total_q * p.num_q_heads;
  if (rows == 0) return cudaSuccess;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > (long long)sms * 16) blocks = (long long)sms * 16;
  const int out_bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
  if (p.topk <= 32) {
    if (partials_fp32(p))
      return launch_pdl(k_combine_small<float>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, st,
                        (const int32_t*)ix.slot_entry, static_cast<const float*>(part_o), part_lse,
                        static_cast<uint8_t*>(out), lse, p.total_q, p.num_q_heads, p.num_kv_heads, p.topk,
                        out_bf16);
    return launch_pdl(k_combine_small<uint16_t>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, st,
                      (const int32_t*)ix.slot_entry, static_cast<const uint16_t*>(part_o), part_lse,
                      static_cast<uint8_t*>(out), lse, p.total_q, p.num_q_heads, p.num_kv_heads, p.topk, out_bf16);
  }
  if (partials_fp32(p))
    return launch_pdl(k_combine<float>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, st,
                      (const int32_t*)ix.slot_entry, static_cast<const float*>(part_o), part_lse,
                      static_cast<uint8_t*>(out), lse, p.total_q, p.num_q_heads, p.num_kv_heads, p.topk, out_bf16);
  return launch_pdl(k_combine<uint16_t>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, st,
                    (const int32_t*)ix.slot_entry, static_cast<const uint16_t*>(part_o), part_lse,
                    static_cast<uint8_t*>(out), lse, p.total_q, p.num_q_heads, p.num_kv_heads, p.topk, out_bf16);
}

}  // namespace mxsa
