"""Block-sparse KV-outer attention for GB300: thin Python binding of libmxsa.

Argument marshalling only -- every step runs in the library's CUDA kernels;
PyTorch provides device memory and streams.  The entry points mirror the C
ABI in include/mxsa.h (build_index, schedule, plan, kvouter_fwd, combine,
read_status, store_kv, the paged-cache store that writes new tokens' K/V
and index keys into the caches, and select_blocks, the top-k block
selection over those index keys), plus ``kvouter_attention`` with the
call shape of the fw-ai/minimax-kernels README's Quick start and
``SparseAttention`` which keeps the workspaces of one problem shape for
repeated calls.

There is no fallback: the first call into the library raises ImportError
when libmxsa.so has not been built, and every library error is raised as
``MxsaError``.  (The package itself imports without the library so that the
build script and the input generator stay usable.)
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmxsa.so")

BF16, FP16, FP8_E4M3, NVFP4 = 0, 1, 2, 3
_DTYPE_CODE = {torch.bfloat16: BF16, torch.float16: FP16, torch.float8_e4m3fn: FP8_E4M3, "nvfp4": NVFP4}
_CODE_DTYPE = {BF16: torch.bfloat16, FP16: torch.float16, FP8_E4M3: torch.float8_e4m3fn, NVFP4: torch.uint8}
# NVFP4 caches are bytes [pages, Hkv, page_size * NVFP4_ROW_BYTES]: per (page,
# kv head), page_size rows of 64 E2M1 code bytes, then page_size rows of 8
# E4M3 scale bytes (one per 16 elements)
NVFP4_ROW_BYTES = 72

FLAG_NAMES = {1: "SEL_RANGE", 2: "SEL_DUP", 4: "PAGE", 8: "CAUSAL_LEN", 16: "LEN", 32: "TIMEOUT",
              64: "SCHEDULE", 128: "CU"}
STATUS_NAMES = {0: "MXSA_OK", 1: "MXSA_ERR_INVALID_ARG", 2: "MXSA_ERR_UNSUPPORTED", 3: "MXSA_ERR_WORKSPACE",
                4: "MXSA_ERR_CUDA", 5: "MXSA_ERR_DATA"}
EXPORTED = ["mxsa_version", "mxsa_status_string", "mxsa_workspace_size", "mxsa_build_index", "mxsa_schedule",
            "mxsa_plan",
            "mxsa_kvouter_fwd", "mxsa_combine", "mxsa_read_status", "mxsa_index_layout_query",
            "mxsa_sched_layout_query", "mxsa_store_kv", "mxsa_dense_fwd", "mxsa_select_workspace_size",
            "mxsa_select_blocks", "mxsa_dedup_workspace_size", "mxsa_build_index_dedup",
            "mxsa_attention_noalloc", "mxsa_noalloc_read_status"]


class MxsaError(RuntimeError):
    def __init__(self, status: int, what: str, flags: int = 0):
        self.status = status
        self.flags = flags
        names = [n for b, n in FLAG_NAMES.items() if flags & b]
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}" + (f" flags={names}" if names else ""))


class Problem(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_q", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]

    def key(self):
        return tuple(getattr(self, f) for f, _ in self._fields_)


class IndexLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("header", "seq_info", "token_seq", "slot_entry", "bitmap", "kmap",
                                               "counts", "row_ptr", "entries", "active_keys", "active_valid",
                                               "row_nnz", "row_minb", "row_maxb", "cta_sums", "total")] + \
               [(n, ctypes.c_int64) for n in ("keys_cap", "nslots", "bitmap_words_cap", "kmap_bytes_cap",
                                              "tiles_cap")]


class SchedLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("header", "items", "cost_prefix", "cta_ptr", "items_dec",
                                               "cost_prefix_dec", "cta_ptr_dec", "cta_sums", "decode_bits",
                                               "total")] + \
               [(n, ctypes.c_int64) for n in ("items_cap", "tiles_cap")]


def _load_library(path: Optional[str] = None) -> ctypes.CDLL:
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libmxsa is not built ({path} missing); run __graft_entry__.build() or "
                          f"python -m block_sparse_attention_builder_gb300.build")
    lib = ctypes.CDLL(path)
    P, S = ctypes.c_void_p, ctypes.c_size_t
    lib.mxsa_version.restype = ctypes.c_int32
    lib.mxsa_status_string.restype = ctypes.c_char_p
    lib.mxsa_status_string.argtypes = [ctypes.c_int]
    sig = {
        "mxsa_workspace_size": [P, P, P, P],
        "mxsa_build_index": [P, P, P, P, P, S, P],
        "mxsa_schedule": [P, P, S, ctypes.c_int32, P, S, P],
        "mxsa_plan": [P, P, P, P, P, S, ctypes.c_int32, P, S, P],
        "mxsa_kvouter_fwd": [P, P, P, P, P, P, S, P, S, ctypes.c_int32, P, S, P],
        "mxsa_combine": [P, P, S, P, S, P, P, P],
        "mxsa_read_status": [P, P, P],
        "mxsa_index_layout_query": [P, P],
        "mxsa_sched_layout_query": [P, P],
        "mxsa_store_kv": [P, ctypes.c_int64, P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int32, P, P],
        "mxsa_dense_fwd": [P, P, P, P, P, P, P, P, P, P, P],
        "mxsa_select_workspace_size": [P, ctypes.c_int32, P],
        "mxsa_select_blocks": [P, ctypes.c_int32, P, P, P, P, P, P, S, P, P, P],
        "mxsa_dedup_workspace_size": [P, P],
        "mxsa_build_index_dedup": [P, P, P, P, P, P, S, P, S, P],
        "mxsa_attention_noalloc": [P] * 11,
        "mxsa_noalloc_read_status": [P, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = args
    return lib


_lib_handle: Optional[ctypes.CDLL] = None


def library() -> ctypes.CDLL:
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load_library()
    return _lib_handle


class _LazyLib:
    def __getattr__(self, name):
        return getattr(library(), name)


_lib = _LazyLib()


def _check(status: int, what: str):
    if status != 0:
        raise MxsaError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_ELEM_BYTES = {BF16: 2, FP16: 2, FP8_E4M3: 1}
_ROW_BYTES = {BF16: 256, FP16: 256, FP8_E4M3: 128, NVFP4: NVFP4_ROW_BYTES}  # per (position, kv head)


def _need(what: str, name: str, t: Optional[torch.Tensor], nbytes: int):
    """The kernels index every buffer by the problem's shape, and a pointer
    carries no size: a tensor smaller than that shape, or not contiguous,
    is refused here, before the C call (MXSA_ERR_INVALID_ARG).  Only bytes
    are compared, so raw views of a cache (uint8, int16) are accepted."""
    if t is None:
        return
    if not t.is_contiguous():
        raise MxsaError(1, f"{what}: {name} is not contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise MxsaError(1, f"{what}: {name} holds {have} bytes, the problem needs {nbytes}")


def _need_attention(what: str, prob: Problem, q=None, k_cache=None, v_cache=None, block_tables=None,
                    cu_seqlens_q=None, used_kv_lens=None, sel=None, out=None, lse=None):
    qb, kb = _ELEM_BYTES.get(prob.q_dtype, 2), _ELEM_BYTES.get(prob.kv_dtype, 2)
    rows = max(prob.total_q, 0) * max(prob.num_q_heads, 0)
    cache = max(prob.num_pages, 0) * max(prob.num_kv_heads, 0) * max(prob.page_size, 0) * \
        _ROW_BYTES.get(prob.kv_dtype, 256)
    _need(what, "q", q, rows * 128 * qb)
    _need(what, "k_cache", k_cache, cache)
    _need(what, "v_cache", v_cache, cache)
    _need(what, "block_tables", block_tables, max(prob.num_seqs, 0) * max(prob.max_pages_per_seq, 0) * 4)
    _need(what, "cu_seqlens_q", cu_seqlens_q, (max(prob.num_seqs, 0) + 1) * 8)
    _need(what, "used_kv_lens", used_kv_lens, max(prob.num_seqs, 0) * 4)
    _need(what, "selected", sel, max(prob.total_q, 0) * max(prob.num_kv_heads, 0) * max(prob.topk, 0) * 4)
    _need(what, "out", out, rows * 128 * qb)
    _need(what, "lse", lse, rows * 4)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_problem(num_seqs, total_q, num_q_heads, num_kv_heads, topk, page_size, num_pages, max_pages_per_seq,
                 causal=False, softmax_scale=0.0, q_dtype=torch.bfloat16, kv_dtype=None, head_dim=128) -> Problem:
    """kv_dtype: q_dtype (None), torch.float8_e4m3fn, or "nvfp4" (byte caches
    in the NVFP4_ROW_BYTES layout)."""
    kv_dtype = q_dtype if kv_dtype is None else kv_dtype
    return Problem(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, topk, page_size, num_pages,
                   max_pages_per_seq, int(bool(causal)), float(softmax_scale or 0.0), _DTYPE_CODE[q_dtype],
                   _DTYPE_CODE[kv_dtype])


def workspace_size(prob: Problem) -> Tuple[int, int, int]:
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.mxsa_workspace_size(ctypes.byref(prob), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
           "mxsa_workspace_size")
    return a.value, b.value, c.value


def index_layout(prob: Problem) -> IndexLayout:
    L = IndexLayout()
    _check(_lib.mxsa_index_layout_query(ctypes.byref(prob), ctypes.byref(L)), "mxsa_index_layout_query")
    return L


def sched_layout(prob: Problem) -> SchedLayout:
    L = SchedLayout()
    _check(_lib.mxsa_sched_layout_query(ctypes.byref(prob), ctypes.byref(L)), "mxsa_sched_layout_query")
    return L


def build_index(prob, sel, cu_seqlens_q, used_kv_lens, index_ws, stream=None):
    _need_attention("mxsa_build_index", prob, cu_seqlens_q=cu_seqlens_q, used_kv_lens=used_kv_lens, sel=sel)
    _check(_lib.mxsa_build_index(ctypes.byref(prob), _ptr(sel), _ptr(cu_seqlens_q), _ptr(used_kv_lens),
                                 _ptr(index_ws), index_ws.numel() * index_ws.element_size(), _stream(stream)),
           "mxsa_build_index")


def dedup_workspace_size(prob: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mxsa_dedup_workspace_size(ctypes.byref(prob), ctypes.byref(n)), "mxsa_dedup_workspace_size")
    return n.value


def build_index_dedup(prob, sel, cu_seqlens_q, used_kv_lens, block_tables, index_ws, dedup_ws, stream=None):
    """The index keyed by physical block: rows of sequences whose block
    tables share a full block's pages at the same logical block meet in the
    smallest such sequence's key (same workspace as build_index)."""
    _need_attention("mxsa_build_index_dedup", prob, cu_seqlens_q=cu_seqlens_q, used_kv_lens=used_kv_lens, sel=sel,
                    block_tables=block_tables)
    _check(_lib.mxsa_build_index_dedup(ctypes.byref(prob), _ptr(sel), _ptr(cu_seqlens_q), _ptr(used_kv_lens),
                                       _ptr(block_tables), _ptr(index_ws), index_ws.numel() * index_ws.element_size(),
                                       _ptr(dedup_ws), dedup_ws.numel() * dedup_ws.element_size(), _stream(stream)),
           "mxsa_build_index_dedup")


def schedule(prob, index_ws, sched_ws, num_ctas=0, stream=None):
    _check(_lib.mxsa_schedule(ctypes.byref(prob), _ptr(index_ws), index_ws.numel() * index_ws.element_size(),
                              int(num_ctas), _ptr(sched_ws), sched_ws.numel() * sched_ws.element_size(),
                              _stream(stream)), "mxsa_schedule")


def plan(prob, sel, cu_seqlens_q, used_kv_lens, index_ws, sched_ws, num_ctas=0, stream=None):
    """build_index + schedule in one launch (identical workspaces)."""
    _need_attention("mxsa_plan", prob, cu_seqlens_q=cu_seqlens_q, used_kv_lens=used_kv_lens, sel=sel)
    _check(_lib.mxsa_plan(ctypes.byref(prob), _ptr(sel), _ptr(cu_seqlens_q), _ptr(used_kv_lens), _ptr(index_ws),
                          index_ws.numel() * index_ws.element_size(), int(num_ctas), _ptr(sched_ws),
                          sched_ws.numel() * sched_ws.element_size(), _stream(stream)), "mxsa_plan")


def kvouter_fwd(prob, q, k_cache, v_cache, block_tables, index_ws, sched_ws, partial_ws, num_ctas=0, stream=None):
    _need_attention("mxsa_kvouter_fwd", prob, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables)
    _check(_lib.mxsa_kvouter_fwd(ctypes.byref(prob), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 _ptr(index_ws), index_ws.numel() * index_ws.element_size(), _ptr(sched_ws),
                                 sched_ws.numel() * sched_ws.element_size(), int(num_ctas), _ptr(partial_ws),
                                 partial_ws.numel() * partial_ws.element_size(), _stream(stream)),
           "mxsa_kvouter_fwd")


def combine(prob, index_ws, partial_ws, out, lse=None, stream=None):
    _need_attention("mxsa_combine", prob, out=out, lse=lse)
    _check(_lib.mxsa_combine(ctypes.byref(prob), _ptr(index_ws), index_ws.numel() * index_ws.element_size(),
                             _ptr(partial_ws), partial_ws.numel() * partial_ws.element_size(), _ptr(out), _ptr(lse),
                             _stream(stream)), "mxsa_combine")


def dense_fwd(prob, q, k_cache, v_cache, block_tables, cu_seqlens_q, used_kv_lens, out, lse=None, flags=None,
              stream=None):
    """Dense paged attention (every key of each sequence; causal per the
    problem) straight into out [total_q, Hq, 128] and lse [Hq, total_q]."""
    _need_attention("mxsa_dense_fwd", prob, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                    cu_seqlens_q=cu_seqlens_q, used_kv_lens=used_kv_lens, out=out, lse=lse)
    _need("mxsa_dense_fwd", "flags", flags, 4)
    _check(_lib.mxsa_dense_fwd(ctypes.byref(prob), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(cu_seqlens_q), _ptr(used_kv_lens), _ptr(out), _ptr(lse), _ptr(flags),
                               _stream(stream)), "mxsa_dense_fwd")


def store_kv(prob, loc, k, v, k_cache, v_cache, idx_k=None, idx_cache=None, flags=None, stream=None):
    """Paged-cache store: rows of k, v ([n, Hkv, 128], the problem's q dtype)
    and optionally idx_k ([n, idx_heads, idx_dim]) into the caches at slots
    loc (int64 [n], page * page_size + offset; < 0: not stored), cast to the
    caches' dtype (the unscaled e4m3 cast for FP8).  flags: optional int32
    device tensor that receives MXSA_FLAG_PAGE for slots past the cache."""
    n = int(loc.numel())
    ih, idim = (int(idx_k.shape[1]), int(idx_k.shape[2])) if idx_k is not None else (0, 0)
    what = "mxsa_store_kv"
    qb, kb = _ELEM_BYTES.get(prob.q_dtype, 2), _ELEM_BYTES.get(prob.kv_dtype, 2)
    _need(what, "loc", loc, n * 8)
    _need(what, "k", k, n * prob.num_kv_heads * 128 * qb)
    _need(what, "v", v, n * prob.num_kv_heads * 128 * qb)
    _need_attention(what, prob, k_cache=k_cache, v_cache=v_cache)
    _need(what, "idx_k", idx_k, n * ih * idim * qb)
    _need(what, "idx_cache", idx_cache, max(prob.num_pages, 0) * ih * max(prob.page_size, 0) * idim * kb)
    _need(what, "flags", flags, 4)
    _check(_lib.mxsa_store_kv(ctypes.byref(prob), n, _ptr(loc), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                              _ptr(idx_k), _ptr(idx_cache), ih, idim, _ptr(flags), _stream(stream)), "mxsa_store_kv")


def select_workspace_size(prob: Problem, idx_dim: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.mxsa_select_workspace_size(ctypes.byref(prob), int(idx_dim), ctypes.byref(n)),
           "mxsa_select_workspace_size")
    return n.value


def select_blocks(prob, idx_q, idx_cache, block_tables, cu_seqlens_q, used_kv_lens, sel=None, score_ws=None,
                  flags=None, stream=None):
    """Top-k block selection (mxsa_select_blocks): sel int32 [total_q, Hkv,
    topk] from the index queries idx_q [total_q, Hkv, D] and the paged index
    cache [pages, Hkv, page_size, D] (kv dtype, D = 64 or 128).  Returns
    (sel, score_ws)."""
    what = "mxsa_select_blocks"
    D = int(idx_q.shape[-1])
    kb = _ELEM_BYTES.get(prob.kv_dtype, 2)
    nbytes = select_workspace_size(prob, D)
    if score_ws is None:
        score_ws = torch.empty(nbytes, dtype=torch.uint8, device=idx_q.device)
    if sel is None:
        sel = torch.empty(prob.total_q, prob.num_kv_heads, prob.topk, dtype=torch.int32, device=idx_q.device)
    _need(what, "idx_q", idx_q, max(prob.total_q, 0) * max(prob.num_kv_heads, 0) * D * kb)
    _need(what, "idx_cache", idx_cache, max(prob.num_pages, 0) * max(prob.num_kv_heads, 0) *
          max(prob.page_size, 0) * D * kb)
    _need_attention(what, prob, block_tables=block_tables, cu_seqlens_q=cu_seqlens_q, used_kv_lens=used_kv_lens,
                    sel=sel)
    _need(what, "score_ws", score_ws, nbytes)
    _need(what, "flags", flags, 4)
    _check(_lib.mxsa_select_blocks(ctypes.byref(prob), D, _ptr(idx_q), _ptr(idx_cache), _ptr(block_tables),
                                   _ptr(cu_seqlens_q), _ptr(used_kv_lens), _ptr(score_ws),
                                   score_ws.numel() * score_ws.element_size(), _ptr(sel), _ptr(flags),
                                   _stream(stream)), what)
    return sel, score_ws


def attention_noalloc(prob, q, k_cache, v_cache, sel, block_tables, cu_seqlens_q, used_kv_lens, out, lse=None,
                      stream=None):
    """All four steps with the library's own fixed scratch array (no
    workspace from the caller); the status word is read with
    noalloc_read_status."""
    _need_attention("mxsa_attention_noalloc", prob, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                    cu_seqlens_q=cu_seqlens_q, used_kv_lens=used_kv_lens, sel=sel, out=out, lse=lse)
    _check(_lib.mxsa_attention_noalloc(ctypes.byref(prob), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sel),
                                       _ptr(block_tables), _ptr(cu_seqlens_q), _ptr(used_kv_lens), _ptr(out),
                                       _ptr(lse), _stream(stream)), "mxsa_attention_noalloc")


def noalloc_read_status(stream=None) -> int:
    flags = ctypes.c_int32(0)
    st = _lib.mxsa_noalloc_read_status(_stream(stream), ctypes.byref(flags))
    if st not in (0, 5):
        raise MxsaError(st, "mxsa_noalloc_read_status")
    return flags.value


def read_status(index_ws, stream=None) -> int:
    flags = ctypes.c_int32(0)
    st = _lib.mxsa_read_status(_ptr(index_ws), _stream(stream), ctypes.byref(flags))
    if st not in (0, 5):
        raise MxsaError(st, "mxsa_read_status")
    return flags.value


@dataclass
class Workspaces:
    index: torch.Tensor
    sched: torch.Tensor
    partial: torch.Tensor


def allocate_workspaces(prob: Problem, device) -> Workspaces:
    ib, sb, pb = workspace_size(prob)
    return Workspaces(torch.empty(ib, dtype=torch.uint8, device=device),
                      torch.empty(sb, dtype=torch.uint8, device=device),
                      torch.empty(pb, dtype=torch.uint8, device=device))


class SparseAttention:
    """The four steps for one problem shape, with workspaces kept across calls."""

    def __init__(self, prob: Problem, device="cuda", num_ctas: int = 0, dedup: bool = False):
        self.prob = prob
        self.device = torch.device(device)
        self.ws = allocate_workspaces(prob, self.device)
        self.num_ctas = num_ctas
        # dedup: key the index by physical block (sequences sharing cached
        # prefix pages load each shared block once); needs block_tables
        self.dedup_ws = (torch.empty(dedup_workspace_size(prob), dtype=torch.uint8, device=self.device)
                         if dedup else None)

    def __call__(self, q, k_cache, v_cache, selected, block_tables, cu_seqlens_q, used_kv_lens, out=None,
                 lse=None, return_lse=True, stream=None):
        """All four steps.  out / lse may be pinned host tensors: the combine
        kernel then writes them directly (valid once the stream is synced)."""
        self.prepare(selected, cu_seqlens_q, used_kv_lens, stream, block_tables=block_tables)
        return self.attend(q, k_cache, v_cache, block_tables, out, lse, return_lse, stream)

    def prepare(self, selected, cu_seqlens_q, used_kv_lens, stream=None, block_tables=None):
        """Index + schedule.  The plain index needs only the selections and
        the sequence lengths (one launch), so q and block_tables may still
        be in flight; the dedup index also reads block_tables (two
        launches: the dedup build, then the scheduler)."""
        if self.dedup_ws is None:
            plan(self.prob, selected, cu_seqlens_q, used_kv_lens, self.ws.index, self.ws.sched, self.num_ctas,
                 stream)
            return
        if block_tables is None:
            raise ValueError("the dedup index needs block_tables")
        build_index_dedup(self.prob, selected, cu_seqlens_q, used_kv_lens, block_tables, self.ws.index,
                          self.dedup_ws, stream)
        schedule(self.prob, self.ws.index, self.ws.sched, self.num_ctas, stream)

    def attend(self, q, k_cache, v_cache, block_tables, out=None, lse=None, return_lse=True, stream=None):
        """Forward + combine over the last prepare()'s index and schedule."""
        p = self.prob
        for name, t in (("out", out), ("lse", lse)):
            if t is not None and not t.is_cuda and not t.is_pinned():
                raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
        if out is None:
            out = torch.empty(p.total_q, p.num_q_heads, 128, dtype=q.dtype, device=q.device)
        if return_lse and lse is None:
            lse = torch.empty(p.num_q_heads, p.total_q, dtype=torch.float32, device=q.device)
        kvouter_fwd(p, q, k_cache, v_cache, block_tables, self.ws.index, self.ws.sched, self.ws.partial,
                    self.num_ctas, stream)
        combine(p, self.ws.index, self.ws.partial, out, lse if return_lse else None, stream)
        return out, (lse if return_lse else None)

    def status(self, stream=None) -> int:
        return read_status(self.ws.index, stream)


def kvouter_attention(q, k_cache, v_cache, selected, block_tables, cu_seqlens_q, used_kv_lens, page_size,
                      causal=False, softmax_scale=None, return_lse=False, num_ctas=0, check=True, dedup=False):
    """Block-sparse KV-outer attention with the README Quick-start call shape.

    q [Tq, Hq, 128] bf16/fp16; k_cache/v_cache [pages, Hkv, page_size, 128]
    (q's dtype or float8_e4m3fn), or NVFP4 uint8 [pages, Hkv, page_size * 72]; selected int32 [Tq, Hkv, topk]; block_tables
    int32 [B, max_pages]; cu_seqlens_q int64 [B+1]; used_kv_lens int32 [B].
    Returns (output [Tq, Hq, 128], lse [Hq, Tq] float32 or None).  With
    check=True the device status word is read (one stream sync) and data
    errors are raised.  dedup=True keys the index by physical block, so
    blocks shared through the block tables load once for all sequences.
    """
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("selected", selected),
                    ("block_tables", block_tables), ("cu_seqlens_q", cu_seqlens_q), ("used_kv_lens", used_kv_lens)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if selected.dtype != torch.int32 or block_tables.dtype != torch.int32 or used_kv_lens.dtype != torch.int32:
        raise ValueError("selected, block_tables and used_kv_lens must be int32")
    if cu_seqlens_q.dtype != torch.int64:
        raise ValueError("cu_seqlens_q must be int64")
    Tq, Hq, D = q.shape
    if k_cache.dtype == torch.uint8:  # NVFP4 byte slabs [pages, Hkv, page_size * 72]
        pages, Hkv, row = k_cache.shape
        if k_cache.shape != v_cache.shape or D != 128 or row != page_size * NVFP4_ROW_BYTES:
            raise ValueError("NVFP4 k_cache / v_cache must be [pages, Hkv, page_size * 72] bytes")
        kv_dtype = "nvfp4"
    else:
        pages, Hkv, ps, D2 = k_cache.shape
        if k_cache.shape != v_cache.shape or D2 != D or ps != page_size:
            raise ValueError("k_cache / v_cache shapes disagree with q or page_size")
        kv_dtype = k_cache.dtype
    prob = make_problem(len(used_kv_lens), Tq, Hq, Hkv, selected.shape[2], page_size, pages,
                        block_tables.shape[1], causal, softmax_scale or 0.0, q.dtype, kv_dtype, head_dim=D)
    attn = SparseAttention(prob, q.device, num_ctas, dedup=dedup)
    out, lse = attn(q, k_cache, v_cache, selected, block_tables, cu_seqlens_q, used_kv_lens, return_lse=return_lse)
    if check:
        flags = attn.status()
        if flags:
            raise MxsaError(5, "kvouter_attention", flags)
    return out, lse
