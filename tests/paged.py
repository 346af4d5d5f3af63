"""Test-side construction of paged caches from contiguous per-sequence K/V.

This runs in the opposite direction to the oracle's gather: contiguous
[Hkv, L, 128] tensors are scattered into randomly numbered physical pages, so
a dense reference computed on the contiguous tensors checks the oracle's page
walk independently.
"""
import numpy as np
import torch

from block_sparse_attention_builder_gb300.workloads import TORCH_DTYPE, generate_values, stream_key


def contiguous_kv(seed, lens, hkv, dtype, tensor_id):
    out = []
    for s, L in enumerate(lens):
        n = hkv * L * 128
        v = generate_values(n, stream_key(seed * 31 + s, tensor_id), dtype, "cpu")
        out.append(v.view(hkv, L, 128))
    return out


def scatter_pages(kv_list, ps, rng, extra_pages=3):
    """(cache [pages, Hkv, ps, 128], block_tables [B, maxp]) holding kv_list."""
    hkv = kv_list[0].shape[0]
    dtype = kv_list[0].dtype
    npages = [max(1, (x.shape[1] + ps - 1) // ps) for x in kv_list]
    total = sum(npages) + extra_pages
    perm = rng.permutation(total)
    # filler pages hold finite values so a wrong page walk shows up
    cache = generate_values(total * hkv * ps * 128, 0xABCDEF, _name(dtype), "cpu").view(total, hkv, ps, 128)
    cache = cache.clone()
    bt = np.full((len(kv_list), max(npages)), -1, dtype=np.int32)
    off = 0
    for s, x in enumerate(kv_list):
        L = x.shape[1]
        for lp in range((L + ps - 1) // ps):
            phys = int(perm[off + lp])
            bt[s, lp] = phys
            n = min(ps, L - lp * ps)
            cache[phys, :, :n, :] = x[:, lp * ps: lp * ps + n, :]
        off += npages[s]
    return cache, bt


def _name(dtype):
    for k, v in TORCH_DTYPE.items():
        if v == dtype:
            return k
    raise ValueError(dtype)
