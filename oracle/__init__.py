"""CPU oracle for block-sparse KV-outer attention -- TEST INFRASTRUCTURE ONLY.

A ctypes front end over ``mxsa_oracle.c`` (plain C, IEEE double).  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the product library never does, and shares no code
with it.  See ``mxsa_oracle.c`` for the definitions and their sources.

Functions whose parity is pinned by tests/test_oracle_pins.py:
  attention_rows  -- dense-attention / masked-SDPA / closed-form pins
  combine         -- partition-merge identity against a single softmax
  build_index     -- brute-force per-key scan on small inputs
  build_index_dedup -- brute force over physical block identities; equal to
                     build_index when no pages are shared
  schedule        -- coverage / ordering / balance invariants
  decode          -- every code against torch's own dtype conversions
  encode_e4m3, store -- every bf16/fp16 code against torch's clamp-and-cast
                     (tests/test_store_pins.py)
  encode_e2m1, NVFP4 store and attention -- E2M1 / E4M3 conversions against
                     ml_dtypes, a hand-made layout fixture, attention on
                     NVFP4 caches against the same values in a BF16 cache
                     (tests/test_nvfp4_pins.py)
  select_blocks   -- top-k block selection: exact float64 scores and a
                     brute-force ranking, ties, masks, pages
                     (tests/test_select_pins.py)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp8": 2, "nvfp4": 3}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, pthreads).  With
    MXSA_ORACLE_LIB set, that library is used as it is (the mutant test)."""
    if os.environ.get("MXSA_ORACLE_LIB"):
        return os.environ["MXSA_ORACLE_LIB"]
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_mutant(n: int, out_dir: str) -> str:
    """The oracle with planted mistake n (-DORACLE_MUTANT=n), for the test
    that checks the pins catch it."""
    path = os.path.join(out_dir, f"liboracle_mutant{n}.so")
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", f"-DORACLE_MUTANT={int(n)}",
                           "-o", path, _SRC, "-lm"])
    return path


class OracleProblem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("total_q", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("softmax_scale", ctypes.c_double), ("q_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        _lib.oracle_decode.restype = ctypes.c_double
        _lib.oracle_decode.argtypes = [ctypes.c_int32, ctypes.c_uint32]
        _lib.oracle_attention_rows.restype = ctypes.c_int
        _lib.oracle_attention_rows.argtypes = [P] * 9 + [ctypes.c_int64, P, P, ctypes.c_int32]
        _lib.oracle_combine.restype = None
        _lib.oracle_combine.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P, P]
        _lib.oracle_build_index.restype = ctypes.c_int
        _lib.oracle_build_index.argtypes = [P, P, P, P, P, P, ctypes.c_int64, P, P, P, P]
        _lib.oracle_build_index_dedup.restype = ctypes.c_int
        _lib.oracle_build_index_dedup.argtypes = [P, P, P, P, P, P, P, ctypes.c_int64, P, P, P, P]
        _lib.oracle_block_owners.restype = ctypes.c_int64
        _lib.oracle_block_owners.argtypes = [P, P, P, P, ctypes.c_int64]
        _lib.oracle_encode_e4m3.restype = ctypes.c_uint32
        _lib.oracle_encode_e4m3.argtypes = [ctypes.c_double]
        _lib.oracle_encode_e2m1.restype = ctypes.c_uint32
        _lib.oracle_encode_e2m1.argtypes = [ctypes.c_float]
        _lib.oracle_store.restype = ctypes.c_int64
        _lib.oracle_store.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int64, P, P, P]
        _lib.oracle_select_blocks.restype = ctypes.c_int
        _lib.oracle_select_blocks.argtypes = [P, ctypes.c_int32, P, P, P, P, P, P, P, ctypes.c_int64, P,
                                              ctypes.c_int64, ctypes.c_int32]
        _lib.oracle_schedule.restype = ctypes.c_int
        _lib.oracle_schedule.argtypes = [P, P, P, ctypes.c_int32, P, P, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, P, P, P, P, P, P, ctypes.c_int64, P]
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def problem(num_seqs, total_q, num_q_heads, num_kv_heads, topk, page_size, num_pages, max_pages_per_seq,
            causal, q_dtype="bf16", kv_dtype="bf16", softmax_scale=0.0, head_dim=128) -> OracleProblem:
    return OracleProblem(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, topk, page_size, num_pages,
                         max_pages_per_seq, int(bool(causal)), float(softmax_scale), DTYPE_CODE[q_dtype],
                         DTYPE_CODE[kv_dtype])


def _bits(x) -> np.ndarray:
    """Raw storage bits of a CPU torch tensor (or numpy array) as uint16/uint8."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.element_size() == 1:
                return x.view(torch.uint8).numpy()
            return x.view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def decode(dtype: str, bits: int) -> float:
    return _load().oracle_decode(DTYPE_CODE[dtype], int(bits))


def encode_e4m3(x: float) -> int:
    """The e4m3fn code of x clamped to [-448, 448], nearest value, ties to even."""
    return int(_load().oracle_encode_e4m3(float(x)))


def encode_e2m1(y: float) -> int:
    """The E2M1 code of the single-precision y: nearest value, ties to even,
    saturating at 6, with y's sign."""
    return int(_load().oracle_encode_e2m1(float(y)))


def store(src, loc, cache, page_size: int, src_dtype: str, dst_dtype: str) -> int:
    """Paged-cache store (the write side of the KV cache): rows of `src`
    [n, heads, dim] (bf16/fp16, torch tensor or raw bits) into `cache` (raw
    bits, numpy, updated in place) at slots loc[t] = page * page_size +
    offset; loc < 0 stores nothing.  `cache` is [num_pages, heads,
    page_size, dim], or for dst_dtype "nvfp4" the byte slabs [num_pages,
    heads, page_size * (dim / 2 + dim / 16)].  Returns the number of tokens
    whose slot lies past the cache."""
    lib = _load()
    sb = _c(_bits(src), np.uint16)
    n, heads, dim = (int(v) for v in sb.shape)
    lo = _c(loc, np.int64)
    if dst_dtype == "nvfp4":
        assert cache.flags["C_CONTIGUOUS"] and cache.dtype == np.uint8
        assert cache.shape[1:] == (heads, page_size * (dim // 2 + dim // 16))
    else:
        assert cache.flags["C_CONTIGUOUS"] and cache.shape[1:] == (heads, page_size, dim)
    rc = lib.oracle_store(DTYPE_CODE[src_dtype], DTYPE_CODE[dst_dtype], n, heads, dim, page_size, cache.shape[0],
                          _ptr(lo), _ptr(sb), _ptr(cache))
    if rc < 0:
        raise RuntimeError(f"oracle_store failed: {rc}")
    return int(rc)


def attention_rows(prob: OracleProblem, q, k_cache, v_cache, selected, block_tables, cu_seqlens_q,
                   used_kv_lens, rows: Optional[np.ndarray] = None, nthreads: Optional[int] = None):
    """(out [n, 128] float64, lse [n] float64) for rows t*Hq+h (None: all rows)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    sel = _c(selected, np.int32)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    lens = _c(used_kv_lens, np.int32)
    if rows is not None:
        rows = _c(rows, np.int64)
        n = len(rows)
    else:
        n = prob.total_q * prob.num_q_heads
    out = np.zeros((n, prob.head_dim), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.oracle_attention_rows(ctypes.byref(prob), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(sel), _ptr(bt),
                                   _ptr(cu), _ptr(lens), _ptr(rows) if rows is not None else None,
                                   ctypes.c_int64(n), _ptr(out), _ptr(lse), nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed: {rc}")
    return out, lse


def select_blocks(prob: OracleProblem, dim: int, idx_q, idx_cache, block_tables, cu_seqlens_q, used_kv_lens,
                  with_scores: bool = False, nthreads: Optional[int] = None, rows: Optional[np.ndarray] = None):
    """Top-k block selection (see oracle_select_blocks): sel int32 [Tq, Hkv,
    topk], and with with_scores the block scores float32 [Tq, Hkv, nblk_max]
    (NaN where a block has none).  rows: only these (token * Hkv + kv head)
    rows are computed (the others stay -1 / NaN)."""
    lib = _load()
    qb, kb = _bits(idx_q), _bits(idx_cache)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    lens = _c(used_kv_lens, np.int32)
    T, H, K = prob.total_q, prob.num_kv_heads, prob.topk
    sel = np.full((T, H, K), -1, dtype=np.int32)
    nbm = (prob.max_pages_per_seq * prob.page_size + 127) // 128
    scores = np.full((T, H, nbm), np.nan, dtype=np.float32) if with_scores else None
    rws = None if rows is None else _c(rows, np.int64)
    rc = lib.oracle_select_blocks(ctypes.byref(prob), int(dim), _ptr(qb), _ptr(kb), _ptr(bt), _ptr(cu), _ptr(lens),
                                  _ptr(sel), _ptr(scores) if with_scores else None, ctypes.c_int64(nbm),
                                  _ptr(rws) if rws is not None else None, ctypes.c_int64(0 if rws is None else len(rws)),
                                  int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise RuntimeError(f"oracle_select_blocks failed: {rc}")
    return (sel, scores) if with_scores else sel


def combine(o_parts: np.ndarray, lse_parts: np.ndarray):
    o = _c(o_parts, np.float64)
    lse = _c(lse_parts, np.float64)
    n, d = o.shape
    out = np.zeros(d, dtype=np.float64)
    lse_out = np.zeros(1, dtype=np.float64)
    _load().oracle_combine(n, d, _ptr(o), _ptr(lse), _ptr(out), _ptr(lse_out))
    return out, float(lse_out[0])


def build_index(prob: OracleProblem, selected, cu_seqlens_q, used_kv_lens):
    """Returns dict(nb, row_ptr, entries, slot_entry, flags)."""
    lib = _load()
    sel = _c(selected, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    lens = _c(used_kv_lens, np.int32)
    cap_len = prob.max_pages_per_seq * prob.page_size
    nb_cap = int(sum((min(max(int(L), 0), cap_len) + 127) // 128 for L in lens))
    rp_cap = prob.num_kv_heads * nb_cap + 1
    row_ptr = np.zeros(rp_cap, dtype=np.int32)
    nslots = prob.total_q * prob.num_kv_heads * prob.topk
    entries = np.zeros(max(nslots, 1), dtype=np.int32)
    slot_entry = np.zeros(max(nslots, 1), dtype=np.int32)
    nb = ctypes.c_int32(0)
    nnz = ctypes.c_int32(0)
    flags = ctypes.c_int32(0)
    rc = lib.oracle_build_index(ctypes.byref(prob), _ptr(sel), _ptr(cu), _ptr(lens), ctypes.byref(nb),
                                _ptr(row_ptr), ctypes.c_int64(rp_cap), _ptr(entries), _ptr(slot_entry),
                                ctypes.byref(nnz), ctypes.byref(flags))
    if rc != 0:
        raise RuntimeError(f"oracle_build_index failed: {rc}")
    nkeys = prob.num_kv_heads * nb.value
    return dict(nb=nb.value, row_ptr=row_ptr[:nkeys + 1].copy(), entries=entries[:nnz.value].copy(),
                slot_entry=slot_entry[:nslots].copy(), flags=flags.value)


def build_index_dedup(prob: OracleProblem, selected, cu_seqlens_q, used_kv_lens, block_tables):
    """The index keyed by physical block (cross-sequence dedup): a row's
    selection of a full block whose pages an earlier sequence holds at the
    same logical block joins that sequence's key.  Same dict as build_index."""
    lib = _load()
    sel = _c(selected, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    lens = _c(used_kv_lens, np.int32)
    bt = _c(block_tables, np.int32)
    if bt.shape != (prob.num_seqs, prob.max_pages_per_seq):
        raise ValueError("block_tables must be [num_seqs, max_pages_per_seq]")
    cap_len = prob.max_pages_per_seq * prob.page_size
    nb_cap = int(sum((min(max(int(L), 0), cap_len) + 127) // 128 for L in lens))
    rp_cap = prob.num_kv_heads * nb_cap + 1
    row_ptr = np.zeros(rp_cap, dtype=np.int32)
    nslots = prob.total_q * prob.num_kv_heads * prob.topk
    entries = np.zeros(max(nslots, 1), dtype=np.int32)
    slot_entry = np.zeros(max(nslots, 1), dtype=np.int32)
    nb, nnz, flags = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    rc = lib.oracle_build_index_dedup(ctypes.byref(prob), _ptr(sel), _ptr(cu), _ptr(lens), _ptr(bt),
                                      ctypes.byref(nb), _ptr(row_ptr), ctypes.c_int64(rp_cap), _ptr(entries),
                                      _ptr(slot_entry), ctypes.byref(nnz), ctypes.byref(flags))
    if rc != 0:
        raise RuntimeError(f"oracle_build_index_dedup failed: {rc}")
    nkeys = prob.num_kv_heads * nb.value
    return dict(nb=nb.value, row_ptr=row_ptr[:nkeys + 1].copy(), entries=entries[:nnz.value].copy(),
                slot_entry=slot_entry[:nslots].copy(), flags=flags.value)


def block_owners(prob: OracleProblem, used_kv_lens, block_tables) -> np.ndarray:
    """Owner sequence of every block (cross-sequence dedup), in key order:
    sequence s's blocks at blk_off[s] .. blk_off[s] + ceil(L_s / 128)."""
    lib = _load()
    lens = _c(used_kv_lens, np.int32)
    bt = _c(block_tables, np.int32)
    cap_len = prob.max_pages_per_seq * prob.page_size
    nb_cap = int(sum((min(max(int(L), 0), cap_len) + 127) // 128 for L in lens))
    out = np.zeros(max(nb_cap, 1), dtype=np.int32)
    nb = lib.oracle_block_owners(ctypes.byref(prob), _ptr(lens), _ptr(bt), _ptr(out), ctypes.c_int64(len(out)))
    if nb < 0:
        raise RuntimeError("oracle_block_owners failed")
    return out[:nb].copy()


def schedule(prob: OracleProblem, used_kv_lens, cu_seqlens_q, index: dict, rows_per_item_tiles: int,
             decode_blocks: int, num_ctas: int):
    """Returns dict(items, cost_prefix, cta_ptr) for the normal list and
    dict(items_dec, cost_prefix_dec, cta_ptr_dec) for the decode list."""
    lib = _load()
    lens = _c(used_kv_lens, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    row_ptr = _c(index["row_ptr"], np.int32)
    entries = _c(index["entries"], np.int32) if len(index["entries"]) else np.zeros(1, np.int32)
    cap = max(int(row_ptr[-1]) + 1, 1)
    items_n = np.zeros((cap, 4), dtype=np.int32)
    cost_n = np.zeros(cap + 1, dtype=np.int64)
    cta_n = np.zeros(num_ctas + 1, dtype=np.int32)
    items_d = np.zeros((cap, 4), dtype=np.int32)
    cost_d = np.zeros(cap + 1, dtype=np.int64)
    cta_d = np.zeros(num_ctas + 1, dtype=np.int32)
    counts = np.zeros(2, dtype=np.int64)
    rc = lib.oracle_schedule(ctypes.byref(prob), _ptr(lens), _ptr(cu), index["nb"], _ptr(row_ptr), _ptr(entries),
                             rows_per_item_tiles, decode_blocks, num_ctas, _ptr(items_n), _ptr(cost_n),
                             _ptr(cta_n), _ptr(items_d), _ptr(cost_d), _ptr(cta_d), ctypes.c_int64(cap),
                             _ptr(counts))
    if rc != 0:
        raise RuntimeError("oracle_schedule: item capacity exceeded")
    nn, nd = int(counts[0]), int(counts[1])
    return dict(items=items_n[:nn].copy(), cost_prefix=cost_n[:nn + 1].copy(), cta_ptr=cta_n,
                items_dec=items_d[:nd].copy(), cost_prefix_dec=cost_d[:nd + 1].copy(), cta_ptr_dec=cta_d)


def problem_for(w, softmax_scale: float = 0.0) -> OracleProblem:
    """The oracle problem struct of a generated workload."""
    return problem(w.num_seqs, w.total_q, w.num_q_heads, w.num_kv_heads, w.topk, w.page_size, w.num_pages,
                   w.max_pages_per_seq, w.causal, w.spec.q_dtype, w.spec.kv_dtype, softmax_scale)
