// mxsa_attention_noalloc: the four steps (index, schedule, forward,
// combine) with every workspace placed in one fixed device array that the
// library owns, so the caller never allocates device memory.
//
// Who needs this: code that is not allowed to call cudaMalloc or any
// allocator on its own.  Typical cases are plug-ins living inside a host
// runtime that plans all device memory up front and hands plug-ins only the
// tensors they read and write, and latency-critical loops where a
// cudaMalloc / cudaFree could synchronise the whole device at a bad moment.
// Such a caller passes inputs and outputs only; the scratch lives here.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes, so
// every GPU that loads this library keeps that much memory reserved until
// the process exits.  In host code the array's name is only a host-side
// stand-in, not a device address, so its real address is looked up once per
// device with cudaGetSymbolAddress (with that device current) on the first
// call made on it; make that first call before any stream capture.  All
// calls share the one array: two calls that overlap on the GPU (different
// streams, or different host threads) race on it and must be serialised by
// the caller.  The steps clear everything they need cleared, so contents
// left by an earlier call do no harm.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  The stream must belong to the current device, and the first
// look-up on a device may not happen while the stream is being captured (it
// is a runtime call a capture does not record): both return
// MXSA_ERR_INVALID_ARG before anything runs.
mxsa_status noalloc_scratch_address(cudaStream_t stream, void** out) {
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXSA_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MXSA_ERR_INVALID_ARG;
  const bool capturing = cs != cudaStreamCaptureStatusNone;
  // the stream's device, outside a capture only (a query a capture in its
  // global mode does not allow; a stream being captured was checked when
  // the calls before the capture ran)
  if (stream && !capturing) {
    int sdev = -1;
    if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return MXSA_ERR_INVALID_ARG;
    if (sdev != dev) return MXSA_ERR_INVALID_ARG;  // the array of another device
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    if (capturing) return MXSA_ERR_INVALID_ARG;  // make the first call on a device outside any capture
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return MXSA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return MXSA_OK;
}

}  // namespace

extern "C" mxsa_status mxsa_attention_noalloc(const mxsa_problem* problem, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* sel, const int32_t* block_tables,
                                              const int64_t* cu_seqlens_q, const int32_t* used_kv_lens, void* out,
                                              float* lse, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  size_t ib = 0, sb = 0, pb = 0;
  mxsa_status s = mxsa_workspace_size(problem, &ib, &sb, &pb);
  if (s != MXSA_OK) return s;
  if (ib + sb + pb > kNoAllocScratchBytes) return MXSA_ERR_WORKSPACE;  // problem too large for the fixed array
  void* addr = nullptr;
  s = noalloc_scratch_address(static_cast<cudaStream_t>(stream), &addr);
  if (s != MXSA_OK) return s;
  uint8_t* base = static_cast<uint8_t*>(addr);
  void* index_ws = base;
  void* sched_ws = base + ib;  // ib and sb are multiples of 256 bytes
  void* partial_ws = base + ib + sb;
  s = mxsa_build_index(problem, sel, cu_seqlens_q, used_kv_lens, index_ws, ib, stream);
  if (s != MXSA_OK) return s;
  s = mxsa_schedule(problem, index_ws, ib, 0, sched_ws, sb, stream);
  if (s != MXSA_OK) return s;
  s = mxsa_kvouter_fwd(problem, q, k_cache, v_cache, block_tables, index_ws, ib, sched_ws, sb, 0, partial_ws, pb,
                       stream);
  if (s != MXSA_OK) return s;
  return mxsa_combine(problem, index_ws, ib, partial_ws, pb, out, lse, stream);
}

// The device status word of the last call's index (at the array's start,
// where that call's index workspace begins), as mxsa_read_status reads it
// from a caller's workspace: synchronises `stream` first.
extern "C" mxsa_status mxsa_noalloc_read_status(void* stream, int32_t* device_flags) {
  if (!device_flags) return MXSA_ERR_INVALID_ARG;
  *device_flags = 0;
  void* addr = nullptr;
  const mxsa_status s = noalloc_scratch_address(static_cast<cudaStream_t>(stream), &addr);
  if (s != MXSA_OK) return s;
  return mxsa_read_status(addr, stream, device_flags);
}
