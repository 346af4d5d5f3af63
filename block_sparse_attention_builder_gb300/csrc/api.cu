// C-ABI entry points of libmxsa: argument validation, workspace layout and
// the launches of the four steps (index builder, scheduler, KV-outer
// forward, combine).  Nothing here allocates memory.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "internal.h"

namespace mxsa {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

int64_t max_blocks_per_seq(const mxsa_problem& p) {
  return ((int64_t)p.max_pages_per_seq * p.page_size + 127) / 128;
}

// Shape checks every entry point shares; the dense path and the store take
// the problem without its top-k (they select nothing).
mxsa_status validate_shape(const mxsa_problem& p) {
  if (p.num_seqs < 1 || p.total_q < 0 || p.num_q_heads < 1 || p.num_kv_heads < 1 || p.num_pages < 1 ||
      p.max_pages_per_seq < 1 || (p.causal != 0 && p.causal != 1) || !(p.softmax_scale >= 0.f) ||
      !std::isfinite(p.softmax_scale))
    return MXSA_ERR_INVALID_ARG;
  if (p.num_q_heads % p.num_kv_heads != 0) return MXSA_ERR_INVALID_ARG;
  if (p.head_dim != 128) return MXSA_ERR_UNSUPPORTED;
  if (p.num_q_heads / p.num_kv_heads > 128) return MXSA_ERR_UNSUPPORTED;
  if (p.page_size != 64 && p.page_size != 128) return MXSA_ERR_UNSUPPORTED;
  if (p.q_dtype != MXSA_BF16 && p.q_dtype != MXSA_FP16) return MXSA_ERR_UNSUPPORTED;
  if (p.kv_dtype != p.q_dtype && p.kv_dtype != MXSA_FP8_E4M3 && p.kv_dtype != MXSA_NVFP4)
    return MXSA_ERR_UNSUPPORTED;
  if ((int64_t)p.num_pages * p.num_kv_heads >= (1ll << 31)) return MXSA_ERR_UNSUPPORTED;
  if ((int64_t)p.max_pages_per_seq * p.page_size >= (1ll << 30)) return MXSA_ERR_UNSUPPORTED;
  return MXSA_OK;
}

// The sparse path: the shape plus the top-k and the index's size limits.
mxsa_status validate_problem(const mxsa_problem& p) {
  mxsa_status s = validate_shape(p);
  if (s != MXSA_OK) return s;
  if (p.topk < 1) return MXSA_ERR_INVALID_ARG;
  if (p.topk > 256) return MXSA_ERR_UNSUPPORTED;
  const int64_t nslots = (int64_t)p.total_q * p.num_kv_heads * p.topk;
  if (nslots >= (1ll << 26)) return MXSA_ERR_UNSUPPORTED;  // slot ids and packed scan fields
  const int64_t keys_cap = (int64_t)p.num_kv_heads * p.num_seqs * max_blocks_per_seq(p);
  if (keys_cap >= (1ll << 31) - 1) return MXSA_ERR_UNSUPPORTED;
  return MXSA_OK;
}

mxsa_status index_layout(const mxsa_problem& p, mxsa_index_layout* L) {
  mxsa_status s = validate_problem(p);
  if (s != MXSA_OK) return s;
  std::memset(L, 0, sizeof(*L));
  const int64_t B = p.num_seqs, Tq = p.total_q, Hkv = p.num_kv_heads;
  const int64_t mb = max_blocks_per_seq(p);
  L->keys_cap = Hkv * B * mb;
  L->nslots = Tq * Hkv * p.topk;
  L->bitmap_words_cap = Hkv * mb * ((Tq + 31) / 32 + B);
  L->kmap_bytes_cap = Hkv * mb * Tq;
  L->tiles_cap = (L->keys_cap + kScanTile - 1) / kScanTile;
  const int64_t act = L->keys_cap < L->nslots ? L->keys_cap : L->nslots;
  size_t o = 0;
  L->header = o;       o = align_up(o + kHdrInts * 4);
  L->seq_info = o;     o = align_up(o + (size_t)B * sizeof(SeqInfo));
  L->token_seq = o;    o = align_up(o + (size_t)Tq * 4);
  L->slot_entry = o;   o = align_up(o + (size_t)L->nslots * 4);
  L->bitmap = o;       o = align_up(o + (size_t)L->bitmap_words_cap * 4);
  L->kmap = o;         o = align_up(o + (size_t)L->kmap_bytes_cap);
  L->counts = o;       o = align_up(o + (size_t)L->keys_cap * 4);
  L->row_ptr = o;      o = align_up(o + (size_t)(L->keys_cap + 1) * 4);
  L->entries = o;      o = align_up(o + (size_t)L->nslots * 4);
  L->active_keys = o;  o = align_up(o + (size_t)act * 4);
  L->active_valid = o; o = align_up(o + (size_t)act * 4);
  L->row_nnz = o;      o = align_up(o + (size_t)Tq * Hkv * 4);
  L->row_minb = o;     o = align_up(o + (size_t)Tq * Hkv * 4);
  L->row_maxb = o;     o = align_up(o + (size_t)Tq * Hkv * 4);
  L->cta_sums = o;     o = align_up(o + (size_t)kMaxCoopCtas * 3 * 8);
  L->total = o;
  return MXSA_OK;
}

mxsa_status sched_layout(const mxsa_problem& p, mxsa_sched_layout* L) {
  mxsa_index_layout il;
  mxsa_status s = index_layout(p, &il);
  if (s != MXSA_OK) return s;
  std::memset(L, 0, sizeof(*L));
  L->items_cap = il.nslots > 0 ? il.nslots : 1;
  const int64_t act = il.keys_cap < il.nslots ? il.keys_cap : il.nslots;
  L->tiles_cap = (act + kScanTile - 1) / kScanTile;
  size_t o = 0;
  L->header = o;          o = align_up(o + kSchInts * 4);
  L->items = o;           o = align_up(o + (size_t)L->items_cap * 16);
  L->cost_prefix = o;     o = align_up(o + (size_t)(L->items_cap + 1) * 8);
  L->cta_ptr = o;         o = align_up(o + (size_t)(MXSA_MAX_CTAS + 1) * 4);
  L->items_dec = o;       o = align_up(o + (size_t)L->items_cap * 16);
  L->cost_prefix_dec = o; o = align_up(o + (size_t)(L->items_cap + 1) * 8);
  L->cta_ptr_dec = o;     o = align_up(o + (size_t)(MXSA_MAX_CTAS + 1) * 4);
  L->cta_sums = o;        o = align_up(o + (size_t)kMaxCoopCtas * 16);
  L->decode_bits = o;     o = align_up(o + (size_t)((act + 31) / 32) * 4);
  L->total = o;
  return MXSA_OK;
}

// Partial outputs: one 128-value row per (entry, head), the normalised
// o = O / l of one block or decode run (its values lie within the range of
// the V rows it averages), in FP32 or in the 16-bit q dtype
// (partials_fp32), then one FP32 lse per row.
static void partial_layout(const mxsa_problem& p, size_t* o_off, size_t* lse_off, size_t* total) {
  const int64_t nslots = (int64_t)p.total_q * p.num_kv_heads * p.topk;
  const int64_t G = p.num_q_heads / p.num_kv_heads;
  *o_off = 0;
  *lse_off = align_up((size_t)nslots * G * 128 * (partials_fp32(p) ? 4 : 2));
  *total = align_up(*lse_off + (size_t)nslots * G * 4);
  if (*total == 0) *total = kAlign;
}

IndexPtrs index_ptrs(const mxsa_problem& p, void* ws) {
  mxsa_index_layout L;
  index_layout(p, &L);
  uint8_t* b = static_cast<uint8_t*>(ws);
  IndexPtrs x;
  x.hdr = reinterpret_cast<int32_t*>(b + L.header);
  x.seq = reinterpret_cast<SeqInfo*>(b + L.seq_info);
  x.token_seq = reinterpret_cast<int32_t*>(b + L.token_seq);
  x.slot_entry = reinterpret_cast<int32_t*>(b + L.slot_entry);
  x.bitmap = reinterpret_cast<uint32_t*>(b + L.bitmap);
  x.kmap = b + L.kmap;
  x.counts = reinterpret_cast<int32_t*>(b + L.counts);
  x.row_ptr = reinterpret_cast<int32_t*>(b + L.row_ptr);
  x.entries = reinterpret_cast<int32_t*>(b + L.entries);
  x.active = reinterpret_cast<int32_t*>(b + L.active_keys);
  x.active_valid = reinterpret_cast<int32_t*>(b + L.active_valid);
  x.row_nnz = reinterpret_cast<int32_t*>(b + L.row_nnz);
  x.row_minb = reinterpret_cast<int32_t*>(b + L.row_minb);
  x.row_maxb = reinterpret_cast<int32_t*>(b + L.row_maxb);
  x.cta_sums = reinterpret_cast<unsigned long long*>(b + L.cta_sums);
  return x;
}

SchedPtrs sched_ptrs(const mxsa_problem& p, void* ws) {
  mxsa_sched_layout L;
  sched_layout(p, &L);
  uint8_t* b = static_cast<uint8_t*>(ws);
  SchedPtrs x;
  x.hdr = reinterpret_cast<int32_t*>(b + L.header);
  x.items = reinterpret_cast<int4*>(b + L.items);
  x.cost_prefix = reinterpret_cast<long long*>(b + L.cost_prefix);
  x.cta_ptr = reinterpret_cast<int32_t*>(b + L.cta_ptr);
  x.items_dec = reinterpret_cast<int4*>(b + L.items_dec);
  x.cost_prefix_dec = reinterpret_cast<long long*>(b + L.cost_prefix_dec);
  x.cta_ptr_dec = reinterpret_cast<int32_t*>(b + L.cta_ptr_dec);
  x.cta_sums = reinterpret_cast<unsigned long long*>(b + L.cta_sums);
  x.dk = reinterpret_cast<uint32_t*>(b + L.decode_bits);
  return x;
}

// Dedup scratch: the page array first (8-byte words), then the block
// arrays and the per-key arrays.
namespace {
struct DedupLayout {
  size_t page_min, owner, gsize, own_count, mbeg, mlist, glist, gkeys, total;
};
DedupLayout dedup_layout(const mxsa_problem& p) {
  const int64_t nb_cap = (int64_t)p.num_seqs * max_blocks_per_seq(p);
  const size_t blk = align_up((size_t)nb_cap * 4), key = align_up((size_t)nb_cap * p.num_kv_heads * 4);
  DedupLayout L;
  size_t o = 0;
  L.page_min = o;  o += align_up((size_t)p.num_pages * 8);
  L.owner = o;     o += blk;
  L.gsize = o;     o += blk;
  L.own_count = o; o += key;
  L.mbeg = o;      o += blk;
  L.mlist = o;     o += blk;
  L.glist = o;     o += blk;
  L.gkeys = o;     o += 2 * key;
  L.total = o;
  return L;
}
}  // namespace

size_t dedup_workspace_bytes(const mxsa_problem& p) { return dedup_layout(p).total; }

DedupPtrs dedup_ptrs(const mxsa_problem& p, void* ws) {
  const DedupLayout L = dedup_layout(p);
  uint8_t* b = static_cast<uint8_t*>(ws);
  DedupPtrs d;
  d.page_min = reinterpret_cast<unsigned long long*>(b + L.page_min);
  d.owner = reinterpret_cast<int32_t*>(b + L.owner);
  d.gsize = reinterpret_cast<int32_t*>(b + L.gsize);
  d.own_count = reinterpret_cast<int32_t*>(b + L.own_count);
  d.mbeg = reinterpret_cast<int32_t*>(b + L.mbeg);
  d.mlist = reinterpret_cast<int32_t*>(b + L.mlist);
  d.glist = reinterpret_cast<int32_t*>(b + L.glist);
  d.gkeys = reinterpret_cast<int2*>(b + L.gkeys);
  return d;
}

static mxsa_status resolve_ctas(int32_t num_ctas, int* out) {
  int n = num_ctas;
  if (n == 0) n = sm_count();
  if (n < 1 || n > MXSA_MAX_CTAS) return MXSA_ERR_INVALID_ARG;
  *out = n;
  return MXSA_OK;
}

}  // namespace mxsa

using namespace mxsa;

extern "C" {

int32_t mxsa_version(void) { return (1 << 16) | 0; }

const char* mxsa_status_string(mxsa_status s) {
  switch (s) {
    case MXSA_OK: return "MXSA_OK";
    case MXSA_ERR_INVALID_ARG: return "MXSA_ERR_INVALID_ARG";
    case MXSA_ERR_UNSUPPORTED: return "MXSA_ERR_UNSUPPORTED";
    case MXSA_ERR_WORKSPACE: return "MXSA_ERR_WORKSPACE";
    case MXSA_ERR_CUDA: return "MXSA_ERR_CUDA";
    case MXSA_ERR_DATA: return "MXSA_ERR_DATA";
  }
  return "unknown mxsa_status";
}

mxsa_status mxsa_workspace_size(const mxsa_problem* problem, size_t* index_bytes, size_t* sched_bytes,
                                size_t* partial_bytes) {
  if (!problem || !index_bytes || !sched_bytes || !partial_bytes) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout il;
  mxsa_sched_layout sl;
  mxsa_status s = index_layout(*problem, &il);
  if (s != MXSA_OK) return s;
  sched_layout(*problem, &sl);
  size_t po, pl, pt;
  partial_layout(*problem, &po, &pl, &pt);
  *index_bytes = il.total;
  *sched_bytes = sl.total;
  *partial_bytes = pt;
  return MXSA_OK;
}

mxsa_status mxsa_index_layout_query(const mxsa_problem* problem, mxsa_index_layout* layout) {
  if (!problem || !layout) return MXSA_ERR_INVALID_ARG;
  return index_layout(*problem, layout);
}

mxsa_status mxsa_sched_layout_query(const mxsa_problem* problem, mxsa_sched_layout* layout) {
  if (!problem || !layout) return MXSA_ERR_INVALID_ARG;
  return sched_layout(*problem, layout);
}

mxsa_status mxsa_build_index(const mxsa_problem* problem, const int32_t* sel, const int64_t* cu_seqlens_q,
                             const int32_t* used_kv_lens, void* index_ws, size_t index_bytes, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout L;
  mxsa_status s = index_layout(*problem, &L);
  if (s != MXSA_OK) return s;
  if (!cu_seqlens_q || !used_kv_lens || !index_ws || (problem->total_q > 0 && !sel)) return MXSA_ERR_INVALID_ARG;
  if (!aligned(sel, 4) || !aligned(cu_seqlens_q, 8) || !aligned(used_kv_lens, 4) || !aligned(index_ws, 16))
    return MXSA_ERR_INVALID_ARG;
  if (index_bytes < L.total) return MXSA_ERR_WORKSPACE;
  IndexPtrs ix = index_ptrs(*problem, index_ws);
  cudaError_t e = launch_build_index(*problem, sel, cu_seqlens_q, used_kv_lens, ix, L,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_dedup_workspace_size(const mxsa_problem* problem, size_t* dedup_bytes) {
  if (!problem || !dedup_bytes) return MXSA_ERR_INVALID_ARG;
  mxsa_status s = validate_problem(*problem);
  if (s != MXSA_OK) return s;
  *dedup_bytes = dedup_workspace_bytes(*problem);
  return MXSA_OK;
}

mxsa_status mxsa_build_index_dedup(const mxsa_problem* problem, const int32_t* sel, const int64_t* cu_seqlens_q,
                                   const int32_t* used_kv_lens, const int32_t* block_tables, void* index_ws,
                                   size_t index_bytes, void* dedup_ws, size_t dedup_bytes, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout L;
  mxsa_status s = index_layout(*problem, &L);
  if (s != MXSA_OK) return s;
  if (!cu_seqlens_q || !used_kv_lens || !block_tables || !index_ws || !dedup_ws || (problem->total_q > 0 && !sel))
    return MXSA_ERR_INVALID_ARG;
  if (!aligned(sel, 4) || !aligned(cu_seqlens_q, 8) || !aligned(used_kv_lens, 4) || !aligned(block_tables, 4) ||
      !aligned(index_ws, 16) || !aligned(dedup_ws, 16))
    return MXSA_ERR_INVALID_ARG;
  if (index_bytes < L.total || dedup_bytes < dedup_workspace_bytes(*problem)) return MXSA_ERR_WORKSPACE;
  IndexPtrs ix = index_ptrs(*problem, index_ws);
  DedupPtrs d = dedup_ptrs(*problem, dedup_ws);
  cudaError_t e = launch_build_index_dedup(*problem, sel, cu_seqlens_q, used_kv_lens, block_tables, ix, d,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_schedule(const mxsa_problem* problem, const void* index_ws, size_t index_bytes, int32_t num_ctas,
                          void* sched_ws, size_t sched_bytes, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout il;
  mxsa_sched_layout sl;
  mxsa_status s = index_layout(*problem, &il);
  if (s != MXSA_OK) return s;
  sched_layout(*problem, &sl);
  if (!index_ws || !sched_ws || !aligned(index_ws, 16) || !aligned(sched_ws, 16)) return MXSA_ERR_INVALID_ARG;
  if (index_bytes < il.total || sched_bytes < sl.total) return MXSA_ERR_WORKSPACE;
  int ctas = 0;
  s = resolve_ctas(num_ctas, &ctas);
  if (s != MXSA_OK) return s;
  IndexPtrs ix = index_ptrs(*problem, const_cast<void*>(index_ws));
  SchedPtrs sc = sched_ptrs(*problem, sched_ws);
  cudaError_t e = launch_schedule(*problem, ix, sc, sl, ctas, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_plan(const mxsa_problem* problem, const int32_t* sel, const int64_t* cu_seqlens_q,
                      const int32_t* used_kv_lens, void* index_ws, size_t index_bytes, int32_t num_ctas,
                      void* sched_ws, size_t sched_bytes, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout il;
  mxsa_sched_layout sl;
  mxsa_status s = index_layout(*problem, &il);
  if (s != MXSA_OK) return s;
  sched_layout(*problem, &sl);
  if (!cu_seqlens_q || !used_kv_lens || !index_ws || !sched_ws || (problem->total_q > 0 && !sel))
    return MXSA_ERR_INVALID_ARG;
  if (!aligned(sel, 4) || !aligned(cu_seqlens_q, 8) || !aligned(used_kv_lens, 4) || !aligned(index_ws, 16) ||
      !aligned(sched_ws, 16))
    return MXSA_ERR_INVALID_ARG;
  if (index_bytes < il.total || sched_bytes < sl.total) return MXSA_ERR_WORKSPACE;
  int ctas = 0;
  s = resolve_ctas(num_ctas, &ctas);
  if (s != MXSA_OK) return s;
  IndexPtrs ix = index_ptrs(*problem, index_ws);
  SchedPtrs sc = sched_ptrs(*problem, sched_ws);
  cudaError_t e = launch_plan(*problem, sel, cu_seqlens_q, used_kv_lens, ix, sc, ctas, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_kvouter_fwd(const mxsa_problem* problem, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const void* index_ws, size_t index_bytes,
                             const void* sched_ws, size_t sched_bytes, int32_t num_ctas, void* partial_ws,
                             size_t partial_bytes, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout il;
  mxsa_sched_layout sl;
  mxsa_status s = index_layout(*problem, &il);
  if (s != MXSA_OK) return s;
  sched_layout(*problem, &sl);
  if (!k_cache || !v_cache || !block_tables || !index_ws || !sched_ws || !partial_ws ||
      (problem->total_q > 0 && !q))
    return MXSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_tables, 4) ||
      !aligned(index_ws, 16) || !aligned(sched_ws, 16) || !aligned(partial_ws, 16))
    return MXSA_ERR_INVALID_ARG;
  size_t po, pl, pt;
  partial_layout(*problem, &po, &pl, &pt);
  if (index_bytes < il.total || sched_bytes < sl.total || partial_bytes < pt) return MXSA_ERR_WORKSPACE;
  int ctas = 0;
  s = resolve_ctas(num_ctas, &ctas);
  if (s != MXSA_OK) return s;
  IndexPtrs ix = index_ptrs(*problem, const_cast<void*>(index_ws));
  SchedPtrs sc = sched_ptrs(*problem, const_cast<void*>(sched_ws));
  uint8_t* pb = static_cast<uint8_t*>(partial_ws);
  int detail = 0;
  cudaError_t e = launch_fwd(*problem, q, k_cache, v_cache, block_tables, ix, sc, ctas,
                             pb + po, reinterpret_cast<float*>(pb + pl),
                             static_cast<cudaStream_t>(stream), &detail);
  if (e != cudaSuccess) return detail ? MXSA_ERR_INVALID_ARG : MXSA_ERR_CUDA;
  return MXSA_OK;
}

// Output pointers of the combine: device memory, or pinned host memory that
// the GPU reaches at the same address (unified addressing; on a Grace-
// Blackwell node the kernel's stores then cross NVLink-C2C directly, with no
// device-to-host copy).  Pageable host memory and unknown pointers are
// refused before any launch.
static bool kernel_writable(const void* p) {
  if (!p) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error the query recorded
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

mxsa_status mxsa_combine(const mxsa_problem* problem, const void* index_ws, size_t index_bytes,
                         const void* partial_ws, size_t partial_bytes, void* out, float* lse, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_index_layout il;
  mxsa_status s = index_layout(*problem, &il);
  if (s != MXSA_OK) return s;
  if (!index_ws || !partial_ws || (problem->total_q > 0 && !out)) return MXSA_ERR_INVALID_ARG;
  if (!aligned(index_ws, 16) || !aligned(partial_ws, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return MXSA_ERR_INVALID_ARG;
  if (!kernel_writable(out) || !kernel_writable(lse)) return MXSA_ERR_INVALID_ARG;
  size_t po, pl, pt;
  partial_layout(*problem, &po, &pl, &pt);
  if (index_bytes < il.total || partial_bytes < pt) return MXSA_ERR_WORKSPACE;
  IndexPtrs ix = index_ptrs(*problem, const_cast<void*>(index_ws));
  const uint8_t* pb = static_cast<const uint8_t*>(partial_ws);
  cudaError_t e = launch_combine(*problem, ix, pb + po,
                                 reinterpret_cast<const float*>(pb + pl), out, lse,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_dense_fwd(const mxsa_problem* problem, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int64_t* cu_seqlens_q, const int32_t* used_kv_lens,
                           void* out, float* lse, int32_t* device_flags, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_status s = validate_shape(*problem);
  if (s != MXSA_OK) return s;
  const mxsa_problem& p = *problem;
  if (p.kv_dtype != p.q_dtype || p.num_seqs > 1024) return MXSA_ERR_UNSUPPORTED;
  if (!block_tables || !cu_seqlens_q || !used_kv_lens) return MXSA_ERR_INVALID_ARG;
  if (p.total_q > 0 && (!q || !k_cache || !v_cache || !out)) return MXSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(cu_seqlens_q, 8) || !aligned(used_kv_lens, 4) || !aligned(lse, 4) ||
      !aligned(device_flags, 4))
    return MXSA_ERR_INVALID_ARG;
  if (!kernel_writable(out) || !kernel_writable(lse)) return MXSA_ERR_INVALID_ARG;
  cudaError_t e = launch_dense(p, q, k_cache, v_cache, block_tables, cu_seqlens_q, used_kv_lens, out, lse,
                               device_flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_store_kv(const mxsa_problem* problem, int64_t n_tokens, const int64_t* loc, const void* k,
                          const void* v, void* k_cache, void* v_cache, const void* idx_k, void* idx_cache,
                          int32_t idx_heads, int32_t idx_dim, int32_t* device_flags, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_status s = validate_shape(*problem);
  if (s != MXSA_OK) return s;
  const mxsa_problem& p = *problem;
  if (n_tokens < 0 || (idx_k == nullptr) != (idx_cache == nullptr)) return MXSA_ERR_INVALID_ARG;
  if (p.kv_dtype == MXSA_NVFP4 && idx_k) return MXSA_ERR_UNSUPPORTED;  // index keys stay 16-bit or FP8
  if (idx_k && (idx_heads <= 0 || idx_dim <= 0 || idx_dim % 8 != 0)) return MXSA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!loc || !k || !v || !k_cache || !v_cache)) return MXSA_ERR_INVALID_ARG;
  if (!aligned(loc, 8) || !aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(idx_k, 16) || !aligned(idx_cache, 16) || !aligned(device_flags, 4))
    return MXSA_ERR_INVALID_ARG;
  cudaError_t e = launch_store(p, n_tokens, loc, k, v, k_cache, v_cache, idx_k, idx_cache, idx_heads, idx_dim,
                               device_flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

// Shape checks of the top-k selection: the sparse problem's (topk, sizes)
// plus the selection's own limits.
static mxsa_status validate_select(const mxsa_problem& p, int32_t idx_dim) {
  mxsa_status s = validate_problem(p);
  if (s != MXSA_OK) return s;
  if (idx_dim != 64 && idx_dim != 128) return MXSA_ERR_UNSUPPORTED;
  if (p.kv_dtype == MXSA_NVFP4) return MXSA_ERR_UNSUPPORTED;  // index keys are 16-bit or FP8
  if (p.num_seqs > 1024 || max_blocks_per_seq(p) > 4096) return MXSA_ERR_UNSUPPORTED;
  return MXSA_OK;
}

mxsa_status mxsa_select_workspace_size(const mxsa_problem* problem, int32_t idx_dim, size_t* score_bytes) {
  if (!problem || !score_bytes) return MXSA_ERR_INVALID_ARG;
  mxsa_status s = validate_select(*problem, idx_dim);
  if (s != MXSA_OK) return s;
  *score_bytes = select_workspace_bytes(*problem);
  return MXSA_OK;
}

mxsa_status mxsa_select_blocks(const mxsa_problem* problem, int32_t idx_dim, const void* idx_q,
                               const void* idx_cache, const int32_t* block_tables, const int64_t* cu_seqlens_q,
                               const int32_t* used_kv_lens, void* score_ws, size_t score_bytes, int32_t* sel,
                               int32_t* device_flags, void* stream) {
  if (!problem) return MXSA_ERR_INVALID_ARG;
  mxsa_status s = validate_select(*problem, idx_dim);
  if (s != MXSA_OK) return s;
  const mxsa_problem& p = *problem;
  if (!block_tables || !cu_seqlens_q || !used_kv_lens || !score_ws) return MXSA_ERR_INVALID_ARG;
  if (p.total_q > 0 && (!idx_q || !idx_cache || !sel)) return MXSA_ERR_INVALID_ARG;
  if (!aligned(idx_q, 16) || !aligned(idx_cache, 16) || !aligned(block_tables, 4) || !aligned(cu_seqlens_q, 8) ||
      !aligned(used_kv_lens, 4) || !aligned(score_ws, 16) || !aligned(sel, 4) || !aligned(device_flags, 4))
    return MXSA_ERR_INVALID_ARG;
  if (score_bytes < select_workspace_bytes(p)) return MXSA_ERR_WORKSPACE;
  cudaError_t e = launch_select(p, idx_dim, idx_q, idx_cache, block_tables, cu_seqlens_q, used_kv_lens, score_ws,
                                sel, device_flags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXSA_OK : MXSA_ERR_CUDA;
}

mxsa_status mxsa_read_status(const void* index_ws, void* stream, int32_t* device_flags) {
  if (!index_ws || !device_flags || !aligned(index_ws, 16)) return MXSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t flags = 0;
  if (cudaMemcpyAsync(&flags, static_cast<const uint8_t*>(index_ws) + kHdrFlags * 4, 4, cudaMemcpyDeviceToHost,
                      st) != cudaSuccess)
    return MXSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MXSA_ERR_CUDA;
  *device_flags = flags;
  return flags ? MXSA_ERR_DATA : MXSA_OK;
}

}  // extern "C"
