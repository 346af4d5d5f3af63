"""Pins of the oracle's NVFP4 KV format (CPU only).

The reading: E2M1 codes with one E4M3 scale per 16 elements, stored as a
(page, kv head) slab of code rows then scale rows; the store's scale is
e4m3(amax / 6) and its codes the nearest E2M1 value of x / scale, ties to
even, saturating at 6.  Pinned to:
  - ml_dtypes' E2M1 and E4M3 conversions (every code, a dense grid of
    single-precision values with every midpoint, random groups);
  - a layout fixture worked by hand (tests/golden/nvfp4_layout.json);
  - attention on an NVFP4 cache equal to attention on a BF16 cache holding
    the same values decoded by ml_dtypes (the values are exact in BF16).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

ml = pytest.importorskip("ml_dtypes")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_lib(bits):
    return np.asarray(bits, np.uint8).view(ml.float4_e2m1fn).astype(np.float64)


def test_e2m1_decode_every_code_against_ml_dtypes():
    lib = _e2m1_lib(np.arange(16, dtype=np.uint8))
    got = np.array([oracle.decode("nvfp4", c) for c in range(16)])
    assert np.array_equal(np.signbit(got), np.signbit(lib)) and np.array_equal(np.abs(got), np.abs(lib))


def test_e2m1_encode_grid_against_ml_dtypes():
    """Every single-precision multiple of 1/64 in [-6, 6] (all the midpoints
    are among them) and its two neighbours."""
    base = np.arange(-6 * 64, 6 * 64 + 1, dtype=np.float32) / np.float32(64)
    ys = np.concatenate([base, np.nextafter(base, np.float32(np.inf)), np.nextafter(base, np.float32(-np.inf))])
    ys = ys[np.abs(ys) <= 6]
    lib = ys.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    got = np.array([oracle.encode_e2m1(float(y)) for y in ys], np.uint8)
    assert np.array_equal(got, lib)


def test_e2m1_encode_saturates_past_six():
    assert [oracle.encode_e2m1(v) for v in (6.5, 7.0, 1e30, float("inf"))] == [7] * 4
    assert [oracle.encode_e2m1(v) for v in (-6.5, -1e30, float("-inf"))] == [15] * 3


def _nvfp4_cache(pages, heads, ps, dim):
    return np.zeros((pages, heads, ps * (dim // 2 + dim // 16)), np.uint8)


def test_store_layout_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "nvfp4_layout.json")))
    ps, dim, slot = fx["page_size"], fx["dim"], fx["slot"]
    row = np.tile(np.asarray(fx["row_group"]["values"], np.float32), dim // 16)
    src = torch.from_numpy(row).to(torch.bfloat16).view(1, 1, dim)
    cache = _nvfp4_cache(1, 1, ps, dim)
    assert oracle.store(src, np.array([slot]), cache, ps, "bf16", "nvfp4") == 0
    slab = cache[0, 0]
    o = fx["codes_offset"]
    assert slab[o:o + dim // 2].tolist() == fx["codes_group_bytes"] * (dim // 16)
    s = fx["scales_offset"]
    assert slab[s:s + dim // 16].tolist() == [fx["scale_byte"]] * (dim // 16)
    untouched = np.ones(slab.size, bool)
    untouched[o:o + dim // 2] = False
    untouched[s:s + dim // 16] = False
    assert not slab[untouched].any()


def _expected_group(x32):
    """Scale and codes of one group by ml_dtypes' conversions."""
    finite = x32[~np.isnan(x32)]
    amax = np.float32(np.abs(finite).max()) if finite.size else np.float32(0)
    s = np.float32(min(amax / np.float32(6), np.float32(448)))
    scale = np.array([s], np.float32).astype(ml.float8_e4m3fn)
    sd = np.float32(scale.astype(np.float32)[0])
    if sd == 0:
        return int(scale.view(np.uint8)[0]), np.zeros(16, np.uint8)
    y = (x32 / sd).astype(np.float32)
    y = np.clip(y, -6, 6)
    codes = (y.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF).astype(np.uint8)
    codes[np.isnan(x32)] = 0
    return int(scale.view(np.uint8)[0]), codes


@pytest.mark.parametrize("src_dtype,seed", [("bf16", 0), ("fp16", 1)])
def test_store_random_rows_against_ml_dtypes(src_dtype, seed):
    rng = np.random.default_rng(seed)
    n, heads, dim, ps, pages = 40, 3, 128, 64, 2
    x = rng.standard_normal((n, heads, dim)).astype(np.float32) * rng.choice([1e-3, 0.3, 5.0, 300.0], (n, heads, 1))
    x[0, 0, :16] = 0.0                  # a zero group: scale 0, codes 0
    x[1, 1, 3] = np.nan                 # NaN: code 0, ignored by amax
    x[2, 2, :16] = 1e-4                 # amax / 6 below half the smallest e4m3 subnormal: scale 0
    tdt = torch.bfloat16 if src_dtype == "bf16" else torch.float16
    src = torch.from_numpy(x).to(tdt)
    xs = src.float().numpy()
    loc = rng.permutation(pages * ps)[:n].astype(np.int64)
    loc[5] = -1
    cache = _nvfp4_cache(pages, heads, ps, dim)
    assert oracle.store(src, loc, cache, ps, src_dtype, "nvfp4") == 0
    for t in range(n):
        if loc[t] < 0:
            continue
        page, off = divmod(int(loc[t]), ps)
        for h in range(heads):
            slab = cache[page, h]
            for j in range(dim // 16):
                scale, codes = _expected_group(xs[t, h, 16 * j:16 * j + 16])
                got = slab[off * 64 + 8 * j: off * 64 + 8 * j + 8]
                assert got.tolist() == (codes[0::2] | (codes[1::2] << 4)).tolist(), (t, h, j)
                assert slab[ps * 64 + off * 8 + j] == scale, (t, h, j)


def test_attention_on_nvfp4_equals_bf16_cache_of_the_same_values():
    from block_sparse_attention_builder_gb300 import workloads as W
    w = W.custom("nvfp4_pin", [1, 3, 40], [300, 700, 2100], 16, 2, 64, 5, True, "uniform", 140, kv_dtype="nvfp4")
    kq, vq = w.k_cache(), w.v_cache()
    ps, D = w.page_size, 128

    def widen(c):
        raw = c.numpy().reshape(w.num_pages, w.num_kv_heads, ps * 72)
        codes = raw[:, :, :ps * 64].reshape(w.num_pages, w.num_kv_heads, ps, 64)
        nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(w.num_pages, w.num_kv_heads, ps, D)
        vals = _e2m1_lib(nib)
        sc = raw[:, :, ps * 64:].reshape(w.num_pages, w.num_kv_heads, ps, D // 16)
        svals = sc.view(ml.float8_e4m3fn).astype(np.float64)
        full = vals * np.repeat(svals, 16, axis=-1)
        t = torch.from_numpy(full).to(torch.bfloat16)
        assert np.array_equal(t.double().numpy(), full)  # exact in BF16
        return t

    kb, vb = widen(kq), widen(vq)
    p4 = oracle.problem_for(w)
    pb = oracle.problem_for(w)
    pb.kv_dtype = oracle.DTYPE_CODE["bf16"]
    args = (w.selected, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    o4, l4 = oracle.attention_rows(p4, w.q(), kq, vq, *args)
    ob, lb = oracle.attention_rows(pb, w.q(), kb, vb, *args)
    assert np.isfinite(l4).any()
    assert np.array_equal(o4, ob) and np.array_equal(l4, lb)
