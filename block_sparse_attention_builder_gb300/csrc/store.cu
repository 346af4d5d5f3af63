// Paged-cache store: the write side of the KV cache that the forward reads
// (a sglang pull request on the same pages, "Summary": the fused K/V/index
// store with an unscaled bf16-to-fp8_e4m3 cast; "Verification": bit-exact
// against x.float().clamp(-448, 448).to(torch.float8_e4m3fn)).
//
// Row (t, h) of a source [n][heads][dim] goes to cache[page][h][off][:],
// page = loc[t] / page_size, off = loc[t] % page_size.  K, V and the
// optional index keys are one launch: one thread per 16-byte source chunk
// (8 values) of K and the same chunk of V, then per index-key chunk, so
// consecutive threads read and write consecutive bytes.  Into
// an e4m3 cache the values are converted two at a time with the saturating
// round-to-nearest-even conversion (448 is the largest finite e4m3fn value,
// so saturating equals clamping first); NaN keeps the sign of its source.
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace mxsa {

namespace {

struct StoreArgs {
  const int64_t* loc;      // slots of this launch's tokens
  const uint16_t* src[3];  // K, V, index keys (this launch's first token)
  uint8_t* dst[3];
  int32_t heads[3];
  int32_t row_chunks[3];   // dim / 8
  int32_t rc_shift[3], heads_shift[3];  // log2 of row_chunks / heads when a power of two, else -1
  uint32_t chunks[3];      // tokens * heads * dim / 8 (< 2^31: the host splits the tokens)
  long long slots;         // num_pages * page_size
  int32_t page_shift, fp8, bf16;
  int32_t* flags;          // may be null
};

__device__ __forceinline__ float to_f32(uint16_t bits, int bf16) {
  return bf16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits));
}

// e4m3 codes of two source values (raw 16-bit words b0, b1), b0's in the
// low byte (no NaN among them)
__device__ __forceinline__ uint32_t e4m3x2(uint16_t b0, uint16_t b1, int bf16) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(to_f32(b1, bf16)), "f"(to_f32(b0, bf16)));
  return r;
}

// the same, for a 16-bit word that may be a NaN: the code takes the NaN's
// sign from the source bits (the fp16 -> f32 conversion does not keep it)
__device__ __forceinline__ uint32_t e4m3_nan_aware(uint16_t b, int bf16) {
  const bool nan = (b & 0x7FFFu) > (bf16 ? 0x7F80u : 0x7C00u);
  return nan ? ((b & 0x8000u) ? 0xFFu : 0x7Fu) : (e4m3x2(b, 0, bf16) & 0xFFu);
}

// any NaN among the eight 16-bit values of s
__device__ __forceinline__ bool any_nan(const uint4& s, int bf16) {
  const uint32_t thr = bf16 ? 0x7F807F80u : 0x7C007C00u;
  const uint32_t w[4] = {s.x, s.y, s.z, s.w};
  uint32_t hit = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) hit |= __vcmpgtu2(w[i] & 0x7FFF7FFFu, thr);
  return hit != 0;
}

// one 16-byte source chunk s (8 values) to its destination: 8 e4m3 bytes or
// the 16 bytes themselves
__device__ __forceinline__ void put_chunk(const uint4& s, uint8_t* dst, long long dst_elem, int fp8, int bf16) {
  if (fp8) {
    uint32_t o[2];
    if (!any_nan(s, bf16)) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t x = i ? s.z : s.x, y = i ? s.w : s.y;
        o[i] = e4m3x2((uint16_t)(x & 0xFFFFu), (uint16_t)(x >> 16), bf16) |
               (e4m3x2((uint16_t)(y & 0xFFFFu), (uint16_t)(y >> 16), bf16) << 16);
      }
    } else {
      const uint32_t w4[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        o[i] = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          o[i] |= e4m3_nan_aware((uint16_t)(w4[2 * i + b / 2] >> (16 * (b & 1))), bf16) << (8 * b);
      }
    }
    *reinterpret_cast<uint2*>(dst + dst_elem) = make_uint2(o[0], o[1]);
  } else {
    *reinterpret_cast<uint4*>(dst + 2 * dst_elem) = s;
  }
}

// Units: first the K/V chunks (one thread stores the same chunk of K and of
// V, which share their token, head and destination offset), then the index
// keys' chunks.
__global__ void __launch_bounds__(256) k_store(StoreArgs a) {
  const uint32_t total = a.chunks[0] + a.chunks[2];
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < total; c += stride) {
    const bool kv = c < a.chunks[0];
    const uint32_t cc = kv ? c : c - a.chunks[0];
    // per-tensor fields by select (a runtime index would copy the
    // parameters to local memory)
    const uint32_t rc = (uint32_t)(kv ? a.row_chunks[0] : a.row_chunks[2]);
    const uint32_t heads = (uint32_t)(kv ? a.heads[0] : a.heads[2]);
    const int rcs = kv ? a.rc_shift[0] : a.rc_shift[2];
    const int hs = kv ? a.heads_shift[0] : a.heads_shift[2];
    const uint32_t row = rcs >= 0 ? cc >> rcs : cc / rc, part = cc - row * rc;
    const uint32_t t = hs >= 0 ? row >> hs : row / heads, h = row - t * heads;
    const long long l = __ldg(a.loc + t);
    if (l < 0) continue;  // the token is not stored
    if (l >= a.slots) {
      if (a.flags && kv && h == 0 && part == 0) atomicOr(a.flags, MXSA_FLAG_PAGE);
      continue;
    }
    const long long page = l >> a.page_shift, off = l & ((1LL << a.page_shift) - 1);
    const long long dst_elem = ((page * heads + h) << a.page_shift | off) * (8LL * rc) + 8LL * part;
    if (kv) {
      const uint4 sk = __ldcs(reinterpret_cast<const uint4*>(a.src[0]) + cc);
      const uint4 sv = __ldcs(reinterpret_cast<const uint4*>(a.src[1]) + cc);
      put_chunk(sk, a.dst[0], dst_elem, a.fp8, a.bf16);
      put_chunk(sv, a.dst[1], dst_elem, a.fp8, a.bf16);
    } else {
      put_chunk(__ldcs(reinterpret_cast<const uint4*>(a.src[2]) + cc), a.dst[2], dst_elem, a.fp8, a.bf16);
    }
  }
}

// ------------------------------------------------------------------ NVFP4
// The NVFP4 cache (E2M1 codes, one E4M3 scale per 16 elements; the MSA
// summary page lists the format, the layout and scaling are this library's):
// a (page, head) slab holds page_size rows of 64 code bytes (element 2i in
// the low nibble of byte i) and then page_size rows of 8 scale bytes.  A
// group of 16 values x stores scale = e4m3(amax / 6) (single-precision
// division, the FP8 cast above) and, with sd the scale's value, codes
// nearest(x / sd) over the E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, ties
// to the even code, saturating at 6, with the quotient's sign; NaN elements
// (which amax ignores) and groups whose scale is 0 store code 0.

// E2M1 code of y: the comparisons put each tie on the even magnitude index
// (0.25 -> 0, 0.75 and 1.25 -> 1.0, 1.75 and 2.5 -> 2, 3.5 and 5 -> 4)
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const uint32_t sign = (__float_as_uint(y) >> 31) << 3;
  const float a = fabsf(y);
  uint32_t i;
  if (a <= 0.25f) i = 0;
  else if (a < 0.75f) i = 1;
  else if (a <= 1.25f) i = 2;
  else if (a < 1.75f) i = 3;
  else if (a <= 2.5f) i = 4;
  else if (a < 3.5f) i = 5;
  else if (a <= 5.0f) i = 6;
  else i = 7;
  return sign | i;
}

struct StoreFp4Args {
  const int64_t* loc;
  const uint16_t* src[2];  // K, V of this launch's first token
  uint8_t* dst[2];
  int32_t heads, heads_shift, page_shift, bf16;
  uint32_t groups;         // tokens * heads * 8
  long long slots;
  int32_t* flags;
};

// one group: its 8 code bytes and its scale byte
__device__ __forceinline__ void put_group_fp4(const uint16_t* src, uint8_t* codes, uint8_t* scale, int bf16) {
  const uint4 s0 = __ldcs(reinterpret_cast<const uint4*>(src));
  const uint4 s1 = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
  const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = to_f32((uint16_t)(w[i] & 0xFFFFu), bf16);
    x[2 * i + 1] = to_f32((uint16_t)(w[i] >> 16), bf16);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));  // fmaxf drops a NaN operand
  uint16_t sc;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(sc) : "f"(0.f), "f"(__fdiv_rn(amax, 6.f)));
  sc &= 0xFFu;
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(sc));
  const float sd = __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t c = (sd == 0.f || isnan(x[i])) ? 0u : e2m1_code(__fdiv_rn(x[i], sd));
    if (i < 8) lo |= c << (4 * i);
    else hi |= c << (4 * (i - 8));
  }
  *reinterpret_cast<uint2*>(codes) = make_uint2(lo, hi);
  *scale = (uint8_t)sc;
}

__global__ void __launch_bounds__(256) k_store_fp4(StoreFp4Args a) {
  const uint32_t stride = gridDim.x * blockDim.x;
  const int ps = 1 << a.page_shift;
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < a.groups; g += stride) {
    const uint32_t row = g >> 3, j = g & 7;  // row = t * heads + h
    const uint32_t t = a.heads_shift >= 0 ? row >> a.heads_shift : row / (uint32_t)a.heads;
    const uint32_t h = row - t * (uint32_t)a.heads;
    const long long l = __ldg(a.loc + t);
    if (l < 0) continue;
    if (l >= a.slots) {
      if (a.flags && h == 0 && j == 0) atomicOr(a.flags, MXSA_FLAG_PAGE);
      continue;
    }
    const long long page = l >> a.page_shift, off = l & (ps - 1);
    const long long slab = (page * a.heads + h) * (long long)ps * 72;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv)
      put_group_fp4(a.src[kv] + (size_t)g * 16, a.dst[kv] + slab + off * 64 + 8 * j,
                    a.dst[kv] + slab + (long long)ps * 64 + off * 8 + j, a.bf16);
  }
}

}  // namespace

// log2(x) when x is a power of two, else -1
static int log2_exact(int x) {
  if (x <= 0 || (x & (x - 1))) return -1;
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

cudaError_t launch_store(const mxsa_problem& p, long long n, const int64_t* loc, const void* k, const void* v,
                         void* k_cache, void* v_cache, const void* idx_k, void* idx_cache, int idx_heads,
                         int idx_dim, int32_t* flags, cudaStream_t st) {
  const int idx_rc = idx_k ? idx_dim / 8 : 0;
  const long long per_token = 2LL * p.num_kv_heads * 16 + (long long)(idx_k ? idx_heads : 0) * idx_rc;  // chunks
  if (n == 0 || per_token == 0) return cudaSuccess;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (p.kv_dtype == MXSA_NVFP4) {  // (no index keys: the caller checked)
    const long long max_tokens = std::max(1LL, (long long)INT32_MAX / (8LL * p.num_kv_heads));
    for (long long t0 = 0; t0 < n; t0 += max_tokens) {
      const long long m = std::min(max_tokens, n - t0);
      StoreFp4Args a{};
      a.loc = loc + t0;
      a.src[0] = static_cast<const uint16_t*>(k) + t0 * p.num_kv_heads * 128;
      a.src[1] = static_cast<const uint16_t*>(v) + t0 * p.num_kv_heads * 128;
      a.dst[0] = static_cast<uint8_t*>(k_cache);
      a.dst[1] = static_cast<uint8_t*>(v_cache);
      a.heads = p.num_kv_heads;
      a.heads_shift = log2_exact(p.num_kv_heads);
      a.page_shift = p.page_size == 128 ? 7 : 6;
      a.bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
      a.groups = (uint32_t)(m * p.num_kv_heads * 8);
      a.slots = (long long)p.num_pages * p.page_size;
      a.flags = flags;
      long long blocks = ((long long)a.groups + 255) / 256;
      if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
      k_store_fp4<<<(unsigned)blocks, 256, 0, st>>>(a);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  const long long max_tokens = std::max(1LL, (long long)INT32_MAX / per_token);  // 32-bit chunk indices
  for (long long t0 = 0; t0 < n; t0 += max_tokens) {
    const long long m = std::min(max_tokens, n - t0);
    StoreArgs a{};
    a.loc = loc + t0;
    a.src[0] = static_cast<const uint16_t*>(k) + t0 * p.num_kv_heads * 128;
    a.src[1] = static_cast<const uint16_t*>(v) + t0 * p.num_kv_heads * 128;
    a.src[2] = idx_k ? static_cast<const uint16_t*>(idx_k) + t0 * idx_heads * idx_dim : nullptr;
    a.dst[0] = static_cast<uint8_t*>(k_cache);
    a.dst[1] = static_cast<uint8_t*>(v_cache);
    a.dst[2] = static_cast<uint8_t*>(idx_cache);
    a.heads[0] = a.heads[1] = p.num_kv_heads;
    a.heads[2] = idx_k ? idx_heads : 1;
    a.row_chunks[0] = a.row_chunks[1] = 16;
    a.row_chunks[2] = idx_k ? idx_rc : 1;
    for (int i = 0; i < 3; ++i) {
      a.rc_shift[i] = log2_exact(a.row_chunks[i]);
      a.heads_shift[i] = log2_exact(a.heads[i]);
    }
    a.chunks[0] = a.chunks[1] = (uint32_t)(m * p.num_kv_heads * 16);
    a.chunks[2] = idx_k ? (uint32_t)(m * idx_heads * idx_rc) : 0u;
    a.slots = (long long)p.num_pages * p.page_size;
    a.page_shift = p.page_size == 128 ? 7 : 6;
    a.fp8 = p.kv_dtype == MXSA_FP8_E4M3 ? 1 : 0;
    a.bf16 = p.q_dtype == MXSA_BF16 ? 1 : 0;
    a.flags = flags;
    const long long total = (long long)a.chunks[0] + a.chunks[2];  // units: K/V chunk pairs, index chunks
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
    k_store<<<(unsigned)blocks, 256, 0, st>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mxsa
