"""GPU parity of the paged-cache store (mxsa_store_kv) with the oracle's
store: bit-exact caches, for the e4m3 cast over every bf16 and fp16 code
and for plain copies, with index keys in the same launch, slots of -1 and
slots past the cache (flagged).  The oracle's encoder is itself pinned to
torch's cast (tests/test_store_pins.py)."""
import numpy as np
import pytest
import torch

import block_sparse_attention_builder_gb300 as mx
import oracle

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.float8_e4m3fn}


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy() if t.element_size() == 1 else t.view(torch.int16).numpy().view(np.uint16)


def _run(src_dt, dst_dt, n, hkv, ps, pages, codes=None, idx=None, seed=0, extra_loc=()):
    rng = np.random.default_rng(seed)
    if codes is None:
        vals = rng.standard_normal((n, hkv, 128)).astype(np.float32) * 100
        k = torch.from_numpy(vals).to(TDT[src_dt])
        v = torch.from_numpy(vals[::-1].copy()).to(TDT[src_dt])
    else:  # every code of the source format, in a seeded order
        flat = rng.permutation(np.resize(codes, n * hkv * 128)).astype(np.uint16)
        k = torch.from_numpy(flat.view(np.int16).reshape(n, hkv, 128)).view(TDT[src_dt])
        v = torch.from_numpy(flat[::-1].copy().view(np.int16).reshape(n, hkv, 128)).view(TDT[src_dt])
    loc = rng.permutation(pages * ps)[:n].astype(np.int64)
    for i, l in extra_loc:
        loc[i] = l
    prob = mx.make_problem(1, n, hkv, hkv, 1, ps, pages, pages, False, q_dtype=TDT[src_dt], kv_dtype=TDT[dst_dt])
    es = 1 if dst_dt == "fp8" else 2
    fill = 0x5A if es == 1 else 0x1234
    host_k = np.full((pages, hkv, ps, 128), fill, dtype=np.uint8 if es == 1 else np.uint16)
    host_v = host_k.copy()
    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    kc, vc = dev(host_k.copy()), dev(host_v.copy())
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = {}
    if idx is not None:
        ih, idim = idx
        iv = torch.from_numpy(rng.standard_normal((n, ih, idim)).astype(np.float32) * 500).to(TDT[src_dt])
        host_i = np.full((pages, ih, ps, idim), fill, dtype=host_k.dtype)
        ic = dev(host_i.copy())
        args = dict(idx_k=iv.cuda(), idx_cache=ic)
    mx.store_kv(prob, torch.from_numpy(loc).cuda(), k.cuda(), v.cuda(), kc, vc, flags=flags, **args)
    torch.cuda.synchronize()
    bad_k = oracle.store(k, loc, host_k, ps, src_dt, dst_dt)
    oracle.store(v, loc, host_v, ps, src_dt, dst_dt)
    assert np.array_equal(_bits(kc).reshape(host_k.shape), host_k)
    assert np.array_equal(_bits(vc).reshape(host_v.shape), host_v)
    if idx is not None:
        oracle.store(iv, loc, host_i, ps, src_dt, dst_dt)
        assert np.array_equal(_bits(ic).reshape(host_i.shape), host_i)
    assert bool(flags.item() & 4) == (bad_k > 0)
    return bad_k


@pytest.mark.parametrize("src", ["bf16", "fp16"])
def test_e4m3_cast_of_every_code(src):
    # 512 tokens x 8 heads x 128 = 8 copies of all 65536 codes, NaNs and infinities included
    _run(src, "fp8", 512, 8, 64, 9, codes=np.arange(65536), seed=1)


@pytest.mark.parametrize("src,dst,ps", [("bf16", "bf16", 64), ("fp16", "fp16", 128), ("bf16", "fp8", 128)])
def test_store_with_index_keys_skips_and_flags(src, dst, ps):
    n = 300
    extra = [(3, -1), (17, -5), (40, 10 ** 9)]  # not stored, not stored, past the cache (flagged)
    bad = _run(src, dst, n, 4, ps, (n + ps - 1) // ps + 2, idx=(2, 64), seed=2, extra_loc=extra)
    assert bad == 1


def test_store_odd_shapes_take_the_division_paths():
    # 3 kv heads and 24-dim index keys (3 chunks a row): neither is a power
    # of two, so the row and token indices come from divisions
    _run("bf16", "fp8", 77, 3, 64, 3, idx=(3, 24), seed=3)
    _run("fp16", "fp16", 50, 3, 128, 1, idx=(1, 8), seed=4)


def test_no_tokens_is_a_no_op():
    prob = mx.make_problem(1, 1, 8, 8, 1, 64, 2, 2, False, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn)
    kc = torch.zeros(2, 8, 64, 128, dtype=torch.uint8, device="cuda")
    e = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    mx.store_kv(prob, torch.empty(0, dtype=torch.int64, device="cuda"), e, e, kc, kc.clone())
    torch.cuda.synchronize()
    assert int(kc.sum()) == 0
