"""Seeded synthetic inputs for block-sparse KV-outer attention.

This module draws inputs only: sequence lengths, paged-cache page tables,
per-query block selections and the q / k / v values.  It holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.

Element values come from a counter-based generator: element ``i`` of a tensor
is ``TABLE[hash(i) >> 16]`` where ``hash`` is Chris Wellons' 32-bit
"lowbias32" integer mixer and ``TABLE`` holds the 65 536 quantiles
``Phi^-1((j + 0.5) / 65536)`` of the standard normal distribution, rounded
(RNE) to the storage dtype.  That is an N(0, 1) sample at 16-bit resolution.
For FP8-e4m3 the quantiles are first clamped to +-448 and then cast, the
cast rule of the fused K/V store in the sglang MiniMax-M3 pull request
(section "Verification").  Because the generator is integer-only torch code,
any element (or any page of the cache) has the same bits whether it is made
on the CPU or on the GPU, so the full-size caches are generated directly in
HBM while the oracle regenerates only the pages it needs.

The five workloads use the tensor layout of the fw-ai/minimax-kernels README
(section "Quick start": token-major q [Tq, Hq, 128], paged caches
[pages, Hkv, page_size, 128], int32 selections [Tq, Hkv, topk] with -1 for
none, int32 block tables, int64 cu_seqlens_q, int32 used_kv_lens).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np
import torch

HEAD_DIM = 128
BLOCK = 128  # tokens per sparse block

_M32 = 0xFFFFFFFF


# --------------------------------------------------------------------------
# counter-based value generator
# --------------------------------------------------------------------------
def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for int64 x in [0, 2^32) without int64 overflow."""
    lo = (x & 0xFFFF) * c
    hi = ((x >> 16) * (c & 0xFFFF)) & 0xFFFF
    return (lo + (hi << 16)) & _M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _hash_index(idx: torch.Tensor, key: int) -> torch.Tensor:
    lo = idx & _M32
    hi = idx >> 32
    return _lowbias32((lo + _lowbias32(hi ^ key)) & _M32)


_TABLES: Dict[str, torch.Tensor] = {}


def _quantile_table(dtype: str) -> torch.Tensor:
    """65 536 normal quantiles as raw storage bits (int16 or uint8), CPU."""
    if dtype not in _TABLES:
        from scipy.special import ndtri

        u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
        z = torch.from_numpy(ndtri(u).astype(np.float32))
        if dtype == "bf16":
            t = z.to(torch.bfloat16).view(torch.int16)
        elif dtype == "fp16":
            t = z.to(torch.float16).view(torch.int16)
        elif dtype == "fp8":
            t = z.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            raise ValueError(dtype)
        _TABLES[dtype] = t.contiguous()
    return _TABLES[dtype]


TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.float8_e4m3fn, "nvfp4": torch.uint8}

# NVFP4 cache slabs: per (page, kv head), page_size rows of 64 code bytes then
# page_size rows of 8 scale bytes (72 bytes per position)
NVFP4_ROW_BYTES = HEAD_DIM // 2 + HEAD_DIM // 16
NVFP4_SCALE_BASE = 0x18  # e4m3 codes 0x18 .. 0x37: scales 2^-4 .. 15/32


def stream_key(seed: int, tensor_id: int) -> int:
    return (seed * 0x9E3779B1 + tensor_id * 0x85EBCA77 + 0x632BE5AB) & _M32


def generate_values(numel: int, key: int, dtype: str, device, start: int = 0, chunk: int = 1 << 25) -> torch.Tensor:
    """Elements [start, start + numel) of the stream `key`, as a flat tensor of `dtype`."""
    table = _quantile_table(dtype).to(device)
    out = torch.empty(numel, dtype=table.dtype, device=device)
    for c0 in range(0, numel, chunk):
        n = min(chunk, numel - c0)
        idx = torch.arange(start + c0, start + c0 + n, dtype=torch.int64, device=device)
        h = _hash_index(idx, key)
        out[c0:c0 + n] = table[(h >> 16) & 0xFFFF]
        del idx, h
    return out.view(TORCH_DTYPE[dtype])


def nvfp4_bytes_at(idx: torch.Tensor, key: int, page_size: int) -> torch.Tensor:
    """Bytes at the int64 flat indices `idx` of an NVFP4 cache drawn from the
    stream `key`: code bytes uniform over all 256 values (two uniform E2M1
    codes), scale bytes uniform over the 32 E4M3 codes from NVFP4_SCALE_BASE
    (2^-4 up to 15/32).  Raw draws only: no value is quantised."""
    h = (_hash_index(idx, key) >> 16) & 0xFFFF
    in_slab = idx % (page_size * NVFP4_ROW_BYTES)
    scale = in_slab >= page_size * (HEAD_DIM // 2)
    return torch.where(scale, NVFP4_SCALE_BASE + (h & 31), h & 0xFF).to(torch.uint8)


def generate_nvfp4(numel: int, key: int, page_size: int, device, chunk: int = 1 << 25) -> torch.Tensor:
    """The first `numel` bytes of an NVFP4 cache (see nvfp4_bytes_at)."""
    out = torch.empty(numel, dtype=torch.uint8, device=device)
    for c0 in range(0, numel, chunk):
        n = min(chunk, numel - c0)
        idx = torch.arange(c0, c0 + n, dtype=torch.int64, device=device)
        out[c0:c0 + n] = nvfp4_bytes_at(idx, key, page_size)
        del idx
    return out


def generate_at(idx: torch.Tensor, key: int, dtype: str) -> torch.Tensor:
    """Elements at the int64 flat indices `idx` of the stream `key` (raw storage bits)."""
    table = _quantile_table(dtype).to(idx.device)
    return table[(_hash_index(idx, key) >> 16) & 0xFFFF]


# --------------------------------------------------------------------------
# workload specification
# --------------------------------------------------------------------------
@dataclass
class WorkloadSpec:
    name: str
    tq: List[int]                      # new query tokens per sequence
    kv_lens: Callable[[np.random.Generator, int], np.ndarray]
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    topk: int
    causal: bool
    selection: str                     # uniform | uniform_last | zipf_diag | uniform_drop10 | hot_groups | all
    seed: int
    q_dtype: str = "bf16"
    kv_dtype: str = "bf16"
    description: str = ""
    extra: dict = field(default_factory=dict)


def _fixed(lens: Sequence[int]):
    return lambda rng, b: np.asarray(lens, dtype=np.int64)


def _uniform_int(lo: int, hi: int):
    return lambda rng, b: rng.integers(lo, hi, size=b, endpoint=True).astype(np.int64)


def physical_blocks_tokens(w: Workload) -> Dict[str, float]:
    """Unique selected blocks counted by physical identity, as the dedup
    index keys them: a block that is full and whose pages are valid is
    (kv head, logical block, its pages); any other block stays
    (kv head, sequence, block).  Plain bookkeeping over the selection
    array and the block tables."""
    Hkv, ps = w.num_kv_heads, w.page_size
    per_blk = BLOCK // ps
    uniq = set()
    tokens_unique = 0
    for s in range(w.num_seqs):
        L = int(w.used_kv_lens[s])
        nblk = (L + BLOCK - 1) // BLOCK
        t0, t1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
        for t in range(t0, t1):
            pos = L - (t1 - t0) + (t - t0)
            for g in range(Hkv):
                for b in w.selected[t, g]:
                    b = int(b)
                    if not 0 <= b < nblk or (w.causal and BLOCK * b > pos):
                        continue
                    pages = tuple(int(x) for x in w.block_tables[s, b * per_blk:(b + 1) * per_blk])
                    full = BLOCK * b + BLOCK <= L and all(0 <= x < w.num_pages for x in pages)
                    key = (g, b, pages) if full else (g, b, ("seq", s))
                    if key not in uniq:
                        uniq.add(key)
                        tokens_unique += min(BLOCK, L - BLOCK * b)
    return {"unique_blocks": len(uniq), "unique_tokens": tokens_unique}


def _log_uniform_int(lo: int, hi: int):
    def f(rng, b):
        x = rng.uniform(math.log(lo), math.log(hi), size=b)
        return np.clip(np.rint(np.exp(x)), lo, hi).astype(np.int64)
    return f


WORKLOADS: Dict[str, WorkloadSpec] = {
    "tiny_decode": WorkloadSpec(
        name="tiny_decode", tq=[1, 1], kv_lens=_fixed([256, 1024]), num_q_heads=16, num_kv_heads=1,
        page_size=64, topk=2, causal=False, selection="uniform", seed=1001,
        description="2 seqs, Tq=1, Hq16/Hkv1, L [256,1024], ps64, top-2 uniform, non-causal"),
    "gqa_decode": WorkloadSpec(
        name="gqa_decode", tq=[1] * 64, kv_lens=_uniform_int(4096, 32768), num_q_heads=64, num_kv_heads=8,
        page_size=64, topk=16, causal=False, selection="uniform_last", seed=1002,
        description="64 seqs, Tq=1, Hq64/Hkv8, L~U[4K,32K], ps64, top-16 incl. last block"),
    "shared_prefill": WorkloadSpec(
        name="shared_prefill", tq=[4096], kv_lens=_fixed([36864]), num_q_heads=16, num_kv_heads=1,
        page_size=128, topk=32, causal=True, selection="zipf_diag", seed=1003,
        description="1 seq, Tq=4096 on 32K context (L=36864), Hq16/Hkv1, ps128, Zipf(1.1) top-31 + diagonal"),
    "fp8_varlen": WorkloadSpec(
        name="fp8_varlen", tq=[1, 1, 1, 1, 8, 8, 64, 64, 256, 256, 512, 512, 1024, 1024, 2048, 2048],
        kv_lens=_uniform_int(2048, 65536), num_q_heads=32, num_kv_heads=4, page_size=128, topk=16,
        causal=True, selection="uniform_drop10", seed=1004, q_dtype="bf16", kv_dtype="fp8",
        description="16 seqs varlen, L~U[2K,64K], Hq32/Hkv4, FP8 K/V, ps128, causal, top-16, 10% -1"),
    "skewed_decode": WorkloadSpec(
        name="skewed_decode", tq=[1] * 256, kv_lens=_log_uniform_int(1024, 262144), num_q_heads=64,
        num_kv_heads=8, page_size=64, topk=64, causal=False, selection="hot_groups", seed=1005,
        description="256 seqs, Tq=1, Hq64/Hkv8, L log-U[1K,256K], ps64, top-64, 8 hot groups"),
}

# Smaller copies of the recipes for profiler captures (a few GB on the device
# at most, unique KV still larger than L2).
WORKLOADS["gqa_decode_p16"] = WorkloadSpec(
    name="gqa_decode_p16", tq=[1] * 16, kv_lens=_uniform_int(4096, 32768), num_q_heads=64, num_kv_heads=8,
    page_size=64, topk=16, causal=False, selection="uniform_last", seed=1012,
    description="profiling copy of gqa_decode with 16 sequences")

# The skewed decode batch read as sequences that share cached prefixes: the
# hot sequences of each group point their first 64 blocks at the group's
# first hot sequence's pages (the cross-sequence dedup case).
WORKLOADS["skewed_decode_shared"] = dataclasses.replace(
    WORKLOADS["skewed_decode"], name="skewed_decode_shared", extra={"shared_prefix_blocks": 64},
    description="skewed_decode with each hot group's first 64 blocks on shared prefix pages")

# Profiling copy of skewed_decode_shared with 64 sequences (4 hot sequences
# per group share their prefix pages).
WORKLOADS["skewed_decode_shared_p64"] = dataclasses.replace(
    WORKLOADS["skewed_decode_shared"], name="skewed_decode_shared_p64", tq=[1] * 64,
    kv_lens=_log_uniform_int(1024, 32768), seed=1015,
    description="profiling copy of skewed_decode_shared: 64 sequences, L log-U[1K, 32K]")

# The GQA decode batch on an NVFP4 cache (E2M1 codes, one E4M3 scale per 16
# elements): 72 bytes per position and kv head against 256 for BF16.
WORKLOADS["gqa_decode_nvfp4"] = dataclasses.replace(
    WORKLOADS["gqa_decode"], name="gqa_decode_nvfp4", kv_dtype="nvfp4",
    description="gqa_decode with NVFP4 K/V (E2M1 + one E4M3 scale per 16 elements)")

# The five workloads, in a fixed order.
WORKLOAD_ORDER = ["tiny_decode", "gqa_decode", "shared_prefill", "fp8_varlen", "skewed_decode"]


# --------------------------------------------------------------------------
# generated workload
# --------------------------------------------------------------------------
@dataclass
class Workload:
    spec: WorkloadSpec
    used_kv_lens: np.ndarray      # int32 [B]
    cu_seqlens_q: np.ndarray      # int64 [B+1]
    block_tables: np.ndarray      # int32 [B, max_pages]  (-1 padded)
    selected: np.ndarray          # int32 [Tq, Hkv, topk]
    num_pages: int

    # shapes -------------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return len(self.used_kv_lens)

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_q_heads(self) -> int:
        return self.spec.num_q_heads

    @property
    def num_kv_heads(self) -> int:
        return self.spec.num_kv_heads

    @property
    def page_size(self) -> int:
        return self.spec.page_size

    @property
    def topk(self) -> int:
        return self.spec.topk

    @property
    def causal(self) -> bool:
        return self.spec.causal

    # values -------------------------------------------------------------
    def q(self, device="cpu") -> torch.Tensor:
        n = self.total_q * self.num_q_heads * HEAD_DIM
        v = generate_values(n, stream_key(self.spec.seed, 1), self.spec.q_dtype, device)
        return v.view(self.total_q, self.num_q_heads, HEAD_DIM)

    def _cache(self, tensor_id: int, device) -> torch.Tensor:
        if self.spec.kv_dtype == "nvfp4":
            n = self.num_pages * self.num_kv_heads * self.page_size * NVFP4_ROW_BYTES
            v = generate_nvfp4(n, stream_key(self.spec.seed, tensor_id), self.page_size, device)
            return v.view(self.num_pages, self.num_kv_heads, self.page_size * NVFP4_ROW_BYTES)
        n = self.num_pages * self.num_kv_heads * self.page_size * HEAD_DIM
        v = generate_values(n, stream_key(self.spec.seed, tensor_id), self.spec.kv_dtype, device)
        return v.view(self.num_pages, self.num_kv_heads, self.page_size, HEAD_DIM)

    def k_cache(self, device="cpu") -> torch.Tensor:
        return self._cache(2, device)

    def v_cache(self, device="cpu") -> torch.Tensor:
        return self._cache(3, device)

    # index tensors of the top-k block selection (one index head per kv head,
    # in the cache dtype): the query side [Tq, Hkv, dim] and the paged index-K
    # cache [pages, Hkv, page_size, dim], paged like K
    def idx_q(self, dim: int, device="cpu") -> torch.Tensor:
        n = self.total_q * self.num_kv_heads * dim
        v = generate_values(n, stream_key(self.spec.seed, 4), self.spec.kv_dtype, device)
        return v.view(self.total_q, self.num_kv_heads, dim)

    def idx_cache(self, dim: int, device="cpu") -> torch.Tensor:
        n = self.num_pages * self.num_kv_heads * self.page_size * dim
        v = generate_values(n, stream_key(self.spec.seed, 5), self.spec.kv_dtype, device)
        return v.view(self.num_pages, self.num_kv_heads, self.page_size, dim)

    def idx_cache_pages(self, dim: int, pages: np.ndarray, device="cpu") -> torch.Tensor:
        """Pages `pages` of the index-K cache as a CPU tensor [n, Hkv, ps, dim]
        (the same values as idx_cache's)."""
        per_page = self.num_kv_heads * self.page_size * dim
        key = stream_key(self.spec.seed, 5)
        pages_t = torch.as_tensor(np.asarray(pages, dtype=np.int64)).to(device)
        ar = torch.arange(per_page, dtype=torch.int64, device=device)
        idx = (pages_t[:, None] * per_page + ar[None, :]).reshape(-1)
        raw = generate_at(idx, key, self.spec.kv_dtype).cpu()
        return raw.view(TORCH_DTYPE[self.spec.kv_dtype]).view(len(pages), self.num_kv_heads, self.page_size, dim)

    def cache_pages(self, tensor_id: int, pages: np.ndarray, device="cpu") -> torch.Tensor:
        """Pages `pages` of the K (2) or V (3) cache as a CPU tensor.  The
        values are generated on `device` (identical bits on any device)."""
        key = stream_key(self.spec.seed, tensor_id)
        if self.spec.kv_dtype == "nvfp4":
            per_page = self.num_kv_heads * self.page_size * NVFP4_ROW_BYTES
            pg = torch.as_tensor(np.asarray(pages, dtype=np.int64)).to(device)
            ar = torch.arange(per_page, dtype=torch.int64, device=device)
            idx = (pg[:, None] * per_page + ar[None, :]).reshape(-1)
            out = nvfp4_bytes_at(idx, key, self.page_size).cpu()
            return out.view(len(pages), self.num_kv_heads, self.page_size * NVFP4_ROW_BYTES)
        per_page = self.num_kv_heads * self.page_size * HEAD_DIM
        pages = torch.as_tensor(np.asarray(pages, dtype=np.int64)).to(device)
        raw = _quantile_table(self.spec.kv_dtype)
        out = torch.empty(len(pages) * per_page, dtype=raw.dtype)
        step = max(1, (1 << 24) // per_page)
        ar = torch.arange(per_page, dtype=torch.int64, device=device)
        for i in range(0, len(pages), step):
            grp = pages[i:i + step]
            idx = (grp[:, None] * per_page + ar[None, :]).reshape(-1)
            out[i * per_page:(i + len(grp)) * per_page] = generate_at(idx, key, self.spec.kv_dtype).cpu()
        return out.view(TORCH_DTYPE[self.spec.kv_dtype]).view(len(pages), self.num_kv_heads, self.page_size,
                                                                 HEAD_DIM)

    def compact_cache_for_rows(self, rows: np.ndarray, device="cpu"):
        """A small cache holding only the pages that rows (flat t*Hq+h) can reach.

        Returns (k_cache, v_cache, block_tables) on the CPU: the physical page
        ids are renumbered 0..n-1 and every page no listed row can reach is
        marked -1 in the returned table.  The values of a kept page are
        identical to the full cache's.
        """
        G = self.num_q_heads // self.num_kv_heads
        ps = self.page_size
        tok = np.asarray(rows) // self.num_q_heads
        g = (np.asarray(rows) % self.num_q_heads) // G
        seq = np.searchsorted(self.cu_seqlens_q, tok, side="right") - 1
        need = {}
        for t, gg, s in zip(tok, g, seq):
            L = int(self.used_kv_lens[s])
            for b in self.selected[t, gg]:
                if b < 0 or b * BLOCK >= L:
                    continue
                first = (b * BLOCK) // ps
                last = (min(b * BLOCK + BLOCK, L) - 1) // ps
                for lp in range(first, last + 1):
                    need[(int(s), lp)] = int(self.block_tables[s, lp])
        phys = np.array(sorted(set(need.values())), dtype=np.int64)
        remap = {int(p): i for i, p in enumerate(phys)}
        bt = np.full_like(self.block_tables, -1)
        for (s, lp), p in need.items():
            bt[s, lp] = remap[p]
        return self.cache_pages(2, phys, device), self.cache_pages(3, phys, device), bt


def _draw_selection(spec: WorkloadSpec, rng: np.random.Generator, lens: np.ndarray, tq: List[int]) -> np.ndarray:
    Hkv, K = spec.num_kv_heads, spec.topk
    total_q = int(sum(tq))
    sel = np.full((total_q, Hkv, K), -1, dtype=np.int32)
    t0 = 0
    for s, (L, n) in enumerate(zip(lens, tq)):
        L = int(L)
        nblk = (L + BLOCK - 1) // BLOCK
        for i in range(n):
            t = t0 + i
            pos = L - n + i
            for g in range(Hkv):
                if spec.selection == "all":
                    row = np.arange(nblk)
                elif spec.selection == "uniform":
                    row = rng.choice(nblk, size=min(K, nblk), replace=False)
                elif spec.selection == "uniform_last":
                    rest = rng.choice(nblk - 1, size=min(K - 1, nblk - 1), replace=False)
                    row = np.concatenate([[nblk - 1], rest])
                elif spec.selection == "zipf_diag":
                    diag = pos // BLOCK
                    w = (np.arange(diag, dtype=np.float64) + 1.0) ** -1.1
                    draws = rng.choice(diag, size=min(K - 1, diag), replace=False, p=w / w.sum())
                    row = np.concatenate([[diag], draws])
                elif spec.selection == "uniform_drop10":
                    nv = (pos // BLOCK + 1) if spec.causal else nblk
                    nv = max(0, min(nv, nblk))
                    row = rng.choice(nv, size=min(K, nv), replace=False) if nv > 0 else np.zeros(0, np.int64)
                elif spec.selection == "hot_groups":
                    grp = s % 8
                    hot = (s // 8) % 2 == 0
                    if hot:
                        perm = np.random.default_rng(spec.seed * 1000 + grp).permutation(64)
                        row = perm[perm < nblk]
                    else:
                        row = rng.choice(nblk, size=min(K, nblk), replace=False)
                else:
                    raise ValueError(spec.selection)
                row = np.asarray(row, dtype=np.int32)[:K]
                sel[t, g, :len(row)] = row
        t0 += n
    if spec.selection == "uniform_drop10":
        drop = rng.random(sel.shape) < 0.10
        sel[drop] = -1
    return sel


def _share_prefix_pages(bt: np.ndarray, lens: np.ndarray, ps: int, prefix_blocks: int) -> None:
    """Shared-prefix page tables (the hot groups of the skewed-decode
    recipe, read as sequences that share a cached prefix): the hot sequences
    of group j (sequence s with s % 8 == j and (s // 8) % 2 == 0) point the
    pages of their first `prefix_blocks` 128-token blocks at the pages of
    the group's first hot sequence, for every block that is full in both.
    The pages they no longer reference stay in the cache, unused."""
    per_blk = BLOCK // ps
    owner: Dict[int, int] = {}
    for s in range(len(lens)):
        if (s // 8) % 2 != 0:
            continue
        j = s % 8
        if j not in owner:
            owner[j] = s
            continue
        o = owner[j]
        full = min(int(lens[s]), int(lens[o])) // BLOCK
        for b in range(min(prefix_blocks, full)):
            bt[s, b * per_blk:(b + 1) * per_blk] = bt[o, b * per_blk:(b + 1) * per_blk]


def make_workload(spec: WorkloadSpec, max_pages_per_seq: Optional[int] = None) -> Workload:
    rng = np.random.default_rng(spec.seed)
    B = len(spec.tq)
    lens = np.asarray(spec.kv_lens(rng, B), dtype=np.int64)
    tq = [int(x) for x in spec.tq]
    ps = spec.page_size
    npages = [(int(L) + ps - 1) // ps for L in lens]
    total_pages = int(sum(npages))
    perm = rng.permutation(total_pages).astype(np.int32)
    maxp = max(npages) if max_pages_per_seq is None else max_pages_per_seq
    maxp = max(maxp, 1)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(npages):
        bt[s, :n] = perm[off:off + n]
        off += n
    if spec.extra.get("shared_prefix_blocks"):
        _share_prefix_pages(bt, lens, ps, int(spec.extra["shared_prefix_blocks"]))
    sel = _draw_selection(spec, rng, lens, tq)
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(tq)
    return Workload(spec=spec, used_kv_lens=lens.astype(np.int32), cu_seqlens_q=cu, block_tables=bt,
                    selected=sel, num_pages=max(total_pages, 1))


def workload(name: str) -> Workload:
    return make_workload(WORKLOADS[name])


def custom(name: str, tq, kv_lens, num_q_heads, num_kv_heads, page_size, topk, causal, selection, seed,
           q_dtype="bf16", kv_dtype="bf16", extra=None) -> Workload:
    """A small workload of the same recipe family, for parity and edge-case tests."""
    spec = WorkloadSpec(name=name, tq=list(tq), kv_lens=_fixed(kv_lens), num_q_heads=num_q_heads,
                        num_kv_heads=num_kv_heads, page_size=page_size, topk=topk, causal=causal,
                        selection=selection, seed=seed, q_dtype=q_dtype, kv_dtype=kv_dtype,
                        extra=dict(extra or {}))
    return make_workload(spec)


def selected_blocks_tokens(w: Workload) -> Dict[str, float]:
    """Counts the sizes the benchmark reports: unique selected (seq, kv-head, block)
    triples with their valid token counts, and the number of block visits.

    Plain bookkeeping over the selection array (no attention arithmetic).
    """
    Hkv = w.num_kv_heads
    uniq = set()
    visits = 0
    tokens_unique = 0
    visit_keys = 0  # sum over (token, kv head, selected block) of the keys the token may use
    for s in range(w.num_seqs):
        L = int(w.used_kv_lens[s])
        nblk = (L + BLOCK - 1) // BLOCK
        t0, t1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
        for t in range(t0, t1):
            pos = L - (t1 - t0) + (t - t0)
            for g in range(Hkv):
                for b in w.selected[t, g]:
                    if 0 <= b < nblk:
                        n_keys = min(BLOCK, L - BLOCK * int(b))
                        if w.causal:
                            n_keys = min(n_keys, pos - BLOCK * int(b) + 1)
                        if n_keys <= 0:
                            continue
                        visits += 1
                        visit_keys += n_keys
                        key = (s, g, int(b))
                        if key not in uniq:
                            uniq.add(key)
                            tokens_unique += min(BLOCK, L - BLOCK * int(b))
    return {"unique_blocks": len(uniq), "unique_tokens": tokens_unique, "block_visits": visits,
            "visit_keys": visit_keys}
