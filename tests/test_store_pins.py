"""Pins of the oracle's paged-cache store (the write side of the KV cache:
the sglang pull request's fused K/V/index store with an unscaled
bf16-to-fp8_e4m3 cast, "Summary" and "Verification").  The e4m3 encoder is
checked against torch's own cast over every bf16 and fp16 code (the exact
expression the pull request verifies against) and against values fixed by
the e4m3fn format definition; the placement against direct indexing."""
import numpy as np
import pytest
import torch

import oracle


def _torch_cast(x: torch.Tensor) -> np.ndarray:
    return x.float().clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_encode_matches_torch_cast_on_every_code(dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(tdt)
    ref = _torch_cast(codes)
    got = np.array([oracle.encode_e4m3(oracle.decode(dtype, c)) for c in range(65536)], dtype=np.uint8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("x,code", [
    (0.0, 0x00), (-0.0, 0x80),
    (1.0, 0x38),                     # E = 7, m = 0
    (448.0, 0x7E), (1e9, 0x7E), (float("inf"), 0x7E), (-1e9, 0xFE),  # largest finite, saturated
    (2.0 ** -9, 0x01), (7 * 2.0 ** -9, 0x07), (2.0 ** -6, 0x08),       # subnormals, smallest normal
    (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),                         # ties to even in the subnormals
    (1.0625, 0x38), (1.1875, 0x3A),  # ties between 1 and 1.125 (even: 1), 1.125 and 1.25 (even: 1.25)
    (15.5 * 2.0 ** -10, 0x08),       # the largest subnormal step rounds up into the normals
    (float("nan"), 0x7F), (-float("nan"), 0xFF),
])
def test_encode_format_points(x, code):
    assert oracle.encode_e4m3(x) == code


@pytest.mark.parametrize("dst", ["bf16", "fp8"])
def test_store_places_rows_by_slot(dst):
    rng = np.random.default_rng(7)
    n, heads, dim, ps, pages = 9, 3, 16, 4, 6
    src = torch.from_numpy(rng.standard_normal((n, heads, dim)).astype(np.float32) * 300).to(torch.bfloat16)
    loc = rng.permutation(pages * ps)[:n].astype(np.int64)
    loc[2] = -1                # no slot: nothing stored
    loc[5] = pages * ps + 3    # past the cache: counted, nothing stored
    sentinel = 0x5A if dst == "fp8" else 0x1234
    cache = np.full((pages, heads, ps, dim), sentinel, dtype=np.uint8 if dst == "fp8" else np.uint16)
    bad = oracle.store(src, loc, cache, ps, "bf16", dst)
    assert bad == 1
    want = np.full_like(cache, sentinel)
    bits = src.view(torch.int16).numpy().view(np.uint16)
    enc = _torch_cast(src)
    for t in range(n):
        if loc[t] < 0 or loc[t] >= pages * ps:
            continue
        page, off = divmod(int(loc[t]), ps)
        want[page, :, off, :] = enc[t] if dst == "fp8" else bits[t]
    assert np.array_equal(cache, want)
