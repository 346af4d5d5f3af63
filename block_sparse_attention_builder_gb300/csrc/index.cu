// Index builder: inverts the query -> block selections into block -> entry
// lists ("index builder" in the test list of the fw-ai/minimax-kernels
// README; the algorithm is this library's).
//
// Keys are (kv head g, sequence s, block b) -> key = g * NB + blk_off[s] + b.
// Within a key the entries are the selection slots (t * Hkv + g) * topk + k
// in increasing token order.  The result is deterministic because the order
// never depends on atomics: each (key, token) pair owns one bit of a per-key
// token bitmap, and the emission walks the set bits in order.
//
// One cooperative launch (all CTAs resident) runs five phases separated by a
// bounded grid barrier:
//   seq    CTA 0: per-sequence scan (L, nblk, block / bitmap / kmap offsets);
//          every CTA: token -> sequence map
//   zero   clears counters, bitmap and scan state
//   mark   one warp per (token, kv head) row: validate, dedupe, set the
//          token's bit in each selected key row, record k
//   reduce the keys are cut into one contiguous chunk per CTA; each CTA
//          sums the entry counts of its chunk
//   scan   each CTA adds the sums of the chunks before it, scans its chunk
//          (row_ptr, the compacted list of keys with entries) and walks the
//          bitmap rows of its keys in order, writing entries[] and the
//          inverse map slot_entry[]
#include <mutex>

#include "index_phases.cuh"

namespace mxsa {

namespace {

using ixp::IndexArgs;
using ixp::kIndexThreads;

__global__ void __launch_bounds__(kIndexThreads) k_index(IndexArgs a) {
  __shared__ unsigned long long tmp[3 * 33];
  __shared__ int32_t rowbuf[ixp::kMarkWarps][256];
  ixp::build_index_phases(a, tmp, rowbuf);
}

}  // namespace

// CTAs of a cooperative launch: at most 2 per SM (all must be resident at
// once); 0 when the device cannot launch cooperatively.  Cached per device.
// Co-resident CTAs of a cooperative launch: the SM count times the CTAs an
// SM holds, at most max_per_sm (more CTAs, more arrivals at each grid
// barrier).  Cached per device and kernel.
int coop_grid(const void* kernel, int threads, int max_per_sm) {
  constexpr int kMaxDev = 64, kMaxKernels = 8;
  static std::mutex mu;
  static const void* keys[kMaxDev][kMaxKernels] = {};
  static int vals[kMaxDev][kMaxKernels] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < kMaxKernels; ++i)
    if (keys[dev][i] == kernel) return vals[dev][i];
  int sms = 0, per_sm = 0, coop = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess) per_sm = 0;
  int g = (coop && sms > 0 && per_sm > 0) ? sms * (per_sm < max_per_sm ? per_sm : max_per_sm) : 0;
  if (g > kMaxCoopCtas) g = kMaxCoopCtas;
  for (int i = 0; i < kMaxKernels; ++i)
    if (!keys[dev][i]) {
      keys[dev][i] = kernel;
      vals[dev][i] = g;
      break;
    }
  return g;
}

cudaError_t launch_build_index(const mxsa_problem& p, const int32_t* sel, const int64_t* cu, const int32_t* lens,
                               const IndexPtrs& ix, const mxsa_index_layout& lay, cudaStream_t st) {
  (void)lay;
  IndexArgs a{ix, sel, cu, lens, p.num_seqs, p.total_q, p.num_kv_heads, p.topk,
              p.max_pages_per_seq * p.page_size, p.causal};
  const int grid = coop_grid(reinterpret_cast<const void*>(k_index), kIndexThreads);
  if (grid <= 0) return cudaErrorNotSupported;
  // header words: flags, sizes, counters and the grid barrier start at zero
  cudaError_t e = cudaMemsetAsync(ix.hdr, 0, kHdrInts * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_index), dim3(grid), dim3(kIndexThreads), args,
                                     0, st);
}

}  // namespace mxsa
