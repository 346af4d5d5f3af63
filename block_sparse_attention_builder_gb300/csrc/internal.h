// Internal declarations shared by the library's translation units:
// workspace layouts, per-sequence metadata and the kernel launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mxsa.h"

namespace mxsa {

// index workspace header (int32 words)
enum : int {
  kHdrFlags = 0,
  kHdrNB = 1,        // blocks over all sequences
  kHdrNnz = 2,       // entries
  kHdrActive = 3,    // keys with at least one entry
  kHdrKeys = 4,      // Hkv * NB
  kHdrBMW = 5,       // bitmap words per kv head
  kHdrKMW = 6,       // kmap bytes per kv head
  kHdrTileCtr = 7,   // dynamic tile counter of the key scan
  kHdrBarCount = 8,  // grid barrier: arrivals (cleared before each launch)
  kHdrAbort = 9,     // grid barrier: set when a barrier wait gave up
  kHdrDedup = 10,    // 1: keys are physical blocks (built by the dedup index build)
  kHdrGroups = 11,   // dedup build: owner blocks with other members (glist)
  kHdrMembers = 12,  // dedup build: member slots handed out (mlist)
  kHdrGroupKeys = 13,  // dedup build: keys of shared owner blocks with entries (gkeys)
  kHdrInts = 16
};

// schedule workspace header (int32 words)
enum : int {
  kSchItems = 0,     // normal (KV-stationary) items
  kSchCtas = 1,
  kSchCostLo = 2,
  kSchCostHi = 3,
  kSchTileCtr = 4,
  kSchDecItems = 5,  // merged decode items
  kSchDecCostLo = 6,
  kSchDecCostHi = 7,
  kSchBarCount = 8,  // grid barrier (as in the index header)
  kSchAbort = 9,
  kSchReserved10 = 10,
  kSchClaim = 11,    // forward: next KV-stationary item to claim (0 after the plan)
  kSchExit = 12,     // forward: CTAs that left (the last one resets both)
  kSchInts = 16
};

// keys of one single-token sequence and kv head are merged into decode items
// of at most this many blocks; decode items need G <= kDecodeMaxG (the rows
// of one token fill one 16-wide MMA N dimension)
constexpr int kDecodeBlocks = 8;
constexpr int kDecodeMaxG = 16;

// Per-sequence metadata written by the index builder.
struct SeqInfo {
  int32_t L;        // used_kv_len clamped to [0, max_pages * page_size]
  int32_t nblk;     // ceil(L / 128)
  int32_t blk_off;  // exclusive prefix of nblk
  int32_t tq;       // new query tokens
  int32_t q_begin;  // cu_seqlens_q[s]
  int32_t bm_off;   // bitmap word offset of the sequence within one kv head
  int32_t km_off;   // kmap byte offset of the sequence within one kv head
  int32_t words;    // ceil(tq / 32): bitmap words per key row
};

struct IndexPtrs {
  int32_t* hdr;
  SeqInfo* seq;
  int32_t* token_seq;
  int32_t* slot_entry;
  uint32_t* bitmap;
  uint8_t* kmap;
  int32_t* counts;
  int32_t* row_ptr;
  int32_t* entries;
  int32_t* active;
  int32_t* active_valid;
  int32_t* row_nnz;                // entries made per (token, kv head) row
  int32_t* row_minb;               // smallest / largest block of those entries
  int32_t* row_maxb;
  unsigned long long* cta_sums;    // per-CTA sums of the cooperative scans (3 per CTA)
};

// CTAs of the cooperative launches (index, schedule) never exceed this
constexpr int kMaxCoopCtas = 1024;
// CTAs of a cooperative launch of `kernel` (index.cu).
int coop_grid(const void* kernel, int threads, int max_per_sm = 2);

struct SchedPtrs {
  int32_t* hdr;
  int4* items;              // normal items {key, entry_begin, n_entries, 0}
  long long* cost_prefix;
  int32_t* cta_ptr;
  int4* items_dec;          // decode items {active_pos, entry, 1, n_keys}
  long long* cost_prefix_dec;
  int32_t* cta_ptr_dec;
  unsigned long long* cta_sums;  // 2 words per CTA: normal, decode
  uint32_t* dk;             // bit a: active key a is a decode key
};

// Scratch of the dedup index build (its own workspace): the smallest packed
// (block, sequence) per physical page, each block's owner sequence, the
// number of blocks each owner block stands for, and each (kv head, block)
// row's own entry count before the rows join their owner's key.
struct DedupPtrs {
  unsigned long long* page_min;  // [num_pages]
  int32_t* owner;                // [blocks]
  int32_t* gsize;                // [blocks]
  int32_t* own_count;            // [Hkv * blocks], key order
  int32_t* mbeg;                 // [blocks]: an owner block's first member in mlist
  int32_t* mlist;                // [blocks]: member sequences of each shared owner block, in order
  int32_t* glist;                // [blocks]: the owner blocks with other members
  int2* gkeys;                   // [Hkv * blocks]: keys of those blocks with entries {key, first entry}
};

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 4;
constexpr int kScanTile = kScanThreads * kScanPerThread;  // keys per look-back tile

// wall-clock limit of every on-device wait (ns); the test build shortens it
#ifndef MXSA_WAIT_LIMIT_NS
#define MXSA_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr unsigned long long kWaitLimitNs = MXSA_WAIT_LIMIT_NS;

int64_t max_blocks_per_seq(const mxsa_problem& p);

// KV blocks stored narrower than q (FP8, NVFP4) are staged and widened to
// q's 16-bit type by the softmax warps before the MMAs.
inline bool kv_widened(const mxsa_problem& p) { return p.kv_dtype == MXSA_FP8_E4M3 || p.kv_dtype == MXSA_NVFP4; }

// Cache kinds: the forward kernels' template parameter.
constexpr int kKind16 = 0, kKindFp8 = 1, kKindFp4 = 2;
inline int cache_kind(const mxsa_problem& p) {
  return p.kv_dtype == MXSA_NVFP4 ? kKindFp4 : (p.kv_dtype == MXSA_FP8_E4M3 ? kKindFp8 : kKind16);
}

// Element type of the partial output rows, per cache kind: the one
// definition behind the kernels' stores, the workspace size and the
// combine's reads.  With 16-bit caches they are stored in the 16-bit q
// dtype, which halves the forward's stores and the combine's reads; with
// widened caches they stay FP32 (there the softmax warps also widen the
// blocks, and the packing on their path costs more than the smaller rows
// save).
__host__ __device__ constexpr bool kind_partials_fp32(int kind) { return kind != kKind16; }
inline bool partials_fp32(const mxsa_problem& p) { return kind_partials_fp32(cache_kind(p)); }
mxsa_status index_layout(const mxsa_problem& p, mxsa_index_layout* L);
mxsa_status sched_layout(const mxsa_problem& p, mxsa_sched_layout* L);
IndexPtrs index_ptrs(const mxsa_problem& p, void* ws);
SchedPtrs sched_ptrs(const mxsa_problem& p, void* ws);
mxsa_status validate_problem(const mxsa_problem& p);

// launchers (return cudaGetLastError())
cudaError_t launch_build_index(const mxsa_problem& p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                               const IndexPtrs& ix, const mxsa_index_layout& lay, cudaStream_t st);
size_t dedup_workspace_bytes(const mxsa_problem& p);
DedupPtrs dedup_ptrs(const mxsa_problem& p, void* ws);
cudaError_t launch_build_index_dedup(const mxsa_problem& p, const int32_t* sel, const int64_t* cu,
                                     const int32_t* lens, const int32_t* block_tables, const IndexPtrs& ix,
                                     const DedupPtrs& d, cudaStream_t st);
cudaError_t launch_plan(const mxsa_problem& p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                        const IndexPtrs& ix, const SchedPtrs& sc, int num_ctas, cudaStream_t st);
cudaError_t launch_schedule(const mxsa_problem& p, const IndexPtrs& ix, const SchedPtrs& sc,
                            const mxsa_sched_layout& lay, int num_ctas, cudaStream_t st);
cudaError_t launch_fwd(const mxsa_problem& p, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const IndexPtrs& ix, const SchedPtrs& sc, int num_ctas,
                       void* part_o, float* part_lse, cudaStream_t st, int* err_detail);
cudaError_t launch_dense(const mxsa_problem& p, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int64_t* cu, const int32_t* lens, void* out, float* lse,
                         int32_t* flags, cudaStream_t st);
cudaError_t launch_store(const mxsa_problem& p, long long n, const int64_t* loc, const void* k, const void* v,
                         void* k_cache, void* v_cache, const void* idx_k, void* idx_cache, int idx_heads,
                         int idx_dim, int32_t* flags, cudaStream_t st);
size_t select_score_bytes(const mxsa_problem& p);
size_t select_workspace_bytes(const mxsa_problem& p);
cudaError_t launch_select(const mxsa_problem& p, int idx_dim, const void* iq, const void* ik, const int32_t* bt,
                          const int64_t* cu, const int32_t* lens, void* ws, int32_t* sel, int32_t* flags,
                          cudaStream_t st);
cudaError_t launch_combine(const mxsa_problem& p, const IndexPtrs& ix, const void* part_o,
                           const float* part_lse, void* out, float* lse, cudaStream_t st);


// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream finishes; it waits for that
// kernel's results with griddepcontrol.wait before reading them.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------------
// device helpers shared by the scan kernels
#ifdef __CUDACC__
// wait until the previous kernel on the stream (a programmatic dependency)
// has completed and its writes are visible; a no-op without one
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// let the next kernel on the stream be scheduled early
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long dev_globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#ifdef MXSA_TEST_HOOKS
// Test builds only (a separate library): CTA g_skip_cta does not arrive at
// the g_skip_barrier-th grid barrier of a launch (1 = the first), so that
// the other CTAs' bounded waits run out.  One copy per translation unit;
// the setter lives beside the kernel it affects.
static __device__ int g_skip_cta = -1;
static __device__ int g_skip_barrier = 0;
#endif

// Grid-wide barrier for kernels launched cooperatively (all CTAs
// co-resident).  bar[0] counts arrivals since the launch and must be 0 at
// launch; the n-th barrier of a launch (n = ++epoch, the same in every CTA)
// completes when it reaches n * nblocks, so no reset or generation word is
// needed and the last arrival releases everyone.  bar[1] is the abort word
// (0 at launch).  The wait is bounded: past the limit it sets
// MXSA_FLAG_TIMEOUT and the abort word, and every later barrier of the
// launch returns at once.  Returns false (in every thread of the CTA) when
// the launch was aborted: the caller must then return instead of starting
// its next phase on data the other CTAs may not have written.
__device__ __forceinline__ bool grid_barrier(int* bar, int* flags, unsigned nblocks, int& epoch) {
  __shared__ int s_ok;
  __syncthreads();
  const int target = ++epoch * (int)nblocks;
  if (threadIdx.x == 0) {
    volatile int* vabort = bar + 1;
    __threadfence();
    int seen;
#ifdef MXSA_TEST_HOOKS
    const bool skip = (int)blockIdx.x == g_skip_cta && epoch == g_skip_barrier;
#else
    constexpr bool skip = false;
#endif
    if (skip)
      seen = -1;  // not counted: this CTA's own wait runs out like the others'
    else
      asm volatile("atom.add.release.gpu.global.s32 %0, [%1], 1;" : "=r"(seen) : "l"(bar) : "memory");
    if (seen + 1 < target) {
      const unsigned long long t0 = dev_globaltimer();
      while (true) {
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(seen) : "l"(bar) : "memory");
        if (seen >= target || *vabort) break;
        if (dev_globaltimer() - t0 > kWaitLimitNs) {
          atomicOr(flags, MXSA_FLAG_TIMEOUT);
          atomicExch(bar + 1, 1);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = *vabort == 0;
  }
  __syncthreads();
  return s_ok != 0;
}

#endif

}  // namespace mxsa
