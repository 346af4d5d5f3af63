"""GPU parity of the NVFP4 KV cache (E2M1 codes with one E4M3 scale per 16
elements): the store's quantisation bit-exact with the oracle's, and the
forward's decode runs and KV-stationary tiles on NVFP4 blocks against the
oracle end to end (BF16/FP16 output atol = rtol = 1e-2, lse 2e-3: the
widened values are exact, so the tolerances are the 16-bit path's)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_builder_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

NUM_SMS = torch.cuda.get_device_properties(0).multi_processor_count

CASES = {
    # decode runs (G = 8, page 64, a partial last block in every row)
    "fp4_decode": W.custom("fp4_decode", [1] * 6, [2100, 2500, 3333, 4096, 4097, 5000], 64, 8, 64, 16, False,
                           "uniform_last", 141, kv_dtype="nvfp4"),
    # KV-stationary tiles, q by TMA (G = 16), page 128, causal diagonal blocks
    "fp4_prefill": W.custom("fp4_prefill", [384], [2432], 16, 1, 128, 8, True, "zipf_diag", 142, kv_dtype="nvfp4"),
    # varlen mix of decode rows and tiles, FP16 q, 10% empty slots
    "fp4_varlen_fp16": W.custom("fp4_varlen_fp16", [1, 8, 64, 130], [300, 1000, 2100, 2900], 32, 4, 128, 6, True,
                                "uniform_drop10", 143, q_dtype="fp16", kv_dtype="nvfp4"),
    # G = 3: the warps' q gather instead of TMA boxes; page 64
    "fp4_gqa3": W.custom("fp4_gqa3", [2, 5, 1], [700, 1300, 129], 12, 4, 64, 5, True, "uniform", 144,
                         kv_dtype="nvfp4"),
    # G = 64 decode rows through the KV-stationary tiles (G > 16)
    "fp4_g64": W.custom("fp4_g64", [1, 3, 20], [200, 900, 1300], 64, 1, 64, 4, True, "uniform", 145,
                        kv_dtype="nvfp4"),
}


@pytest.fixture(scope="module")
def runs():
    return {name: U.run(w) for name, w in CASES.items()}


@pytest.mark.parametrize("name", list(CASES))
def test_nvfp4_end_to_end_matches_oracle(name, runs):
    w = CASES[name]
    attn, out, lse, _ = runs[name]
    assert attn.status() == 0
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, f"{name} out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, f"{name} lse")


@pytest.mark.parametrize("name", ["fp4_prefill", "fp4_varlen_fp16"])
def test_nvfp4_partials_of_normal_items(name, runs):
    """Per-entry partial rows of the KV-stationary items against the
    oracle's attention over each slot's block alone."""
    w = CASES[name]
    attn = runs[name][0]
    G = w.num_q_heads // w.num_kv_heads
    idx = U.read_index(attn)
    sch = U.read_sched(attn, NUM_SMS)
    o_gpu, l_gpu = U.read_partials(attn)
    o_ref, l_ref = U.oracle_slot_partials(w)
    ents = np.concatenate([np.arange(e0, e0 + n) for _, e0, n, _ in sch["items"]])
    slots = idx["entries"][ents]
    rows_gpu = (ents[:, None] * G + np.arange(G)).reshape(-1)
    rows_ref = (slots[:, None] * G + np.arange(G)).reshape(-1)
    U.assert_close_out(o_gpu[rows_gpu], o_ref[rows_ref], 1e-2, f"{name} partial o")
    U.assert_close_lse(l_gpu[rows_gpu], l_ref[rows_ref], 2e-3, f"{name} partial lse")


def test_nvfp4_quickstart_call():
    import block_sparse_attention_builder_gb300 as mx
    w = CASES["fp4_gqa3"]
    inp = U.device_inputs(w)
    out, lse = mx.kvouter_attention(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"],
                                    page_size=w.page_size, causal=True, return_lse=True)
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, "quickstart nvfp4")


@pytest.mark.parametrize("src,ps,seed", [("bf16", 64, 0), ("fp16", 128, 1)])
def test_nvfp4_store_bit_exact(src, ps, seed):
    """Rows of several scales (and a zero group, a NaN, a group whose scale
    rounds to 0, an infinity) quantised by mxsa_store_kv, byte for byte
    against the oracle's store; a slot past the cache is flagged."""
    import block_sparse_attention_builder_gb300 as mx
    rng = np.random.default_rng(seed)
    n, Hkv, pages = 300, 4, 8
    tdt = torch.bfloat16 if src == "bf16" else torch.float16
    x = rng.standard_normal((2, n, Hkv, 128)).astype(np.float32) * \
        rng.choice([1e-3, 0.3, 5.0, 300.0], (2, n, Hkv, 1)).astype(np.float32)
    x[0, 0, 0, :16] = 0.0
    x[1, 1, 1, 5] = np.nan
    x[0, 2, 2, 16:32] = 1e-4
    x[1, 3, 3, 40] = np.inf
    k, v = (torch.from_numpy(x[i]).to(tdt) for i in range(2))
    loc = rng.permutation(pages * ps)[:n].astype(np.int64)
    loc[7] = -1
    loc[9] = pages * ps + 3  # past the cache: flagged, not stored
    prob = mx.make_problem(1, 0, Hkv, Hkv, 1, ps, pages, 1, False, 0.0, tdt, "nvfp4")
    kc = torch.zeros(pages, Hkv, ps * 72, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx.store_kv(prob, torch.from_numpy(loc).cuda(), k.cuda(), v.cuda(), kc, vc, flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & 4
    for src_t, got in ((k, kc), (v, vc)):
        ref = np.zeros((pages, Hkv, ps * 72), np.uint8)
        assert oracle.store(src_t, loc, ref, ps, src, "nvfp4") == 1
        assert np.array_equal(got.cpu().numpy(), ref)


def test_nvfp4_store_then_attend():
    """New tokens stored into an NVFP4 cache by mxsa_store_kv, then attended:
    the output matches the oracle's attention on the oracle-stored cache."""
    import block_sparse_attention_builder_gb300 as mx
    w = CASES["fp4_decode"]
    ps, Hkv = w.page_size, w.num_kv_heads
    inp = U.device_inputs(w)
    kc, vc = inp["k"].clone(), inp["v"].clone()
    # overwrite the last 64 positions of every sequence with stored rows
    locs = []
    for s in range(w.num_seqs):
        L = int(w.used_kv_lens[s])
        for pos in range(L - 64, L):
            locs.append(int(w.block_tables[s, pos // ps]) * ps + pos % ps)
    loc = np.asarray(locs, np.int64)
    rng = np.random.default_rng(7)
    rows = [torch.from_numpy(rng.standard_normal((len(loc), Hkv, 128)).astype(np.float32)).to(torch.bfloat16)
            for _ in range(2)]
    prob = U.problem(w)
    mx.store_kv(prob, torch.from_numpy(loc).cuda(), rows[0].cuda(), rows[1].cuda(), kc, vc)
    attn = mx.SparseAttention(prob, "cuda")
    out, lse = attn(inp["q"], kc, vc, inp["sel"], inp["bt"], inp["cu"], inp["lens"])
    torch.cuda.synchronize()
    k_ref, v_ref = w.k_cache().numpy().copy(), w.v_cache().numpy().copy()
    oracle.store(rows[0], loc, k_ref, ps, "bf16", "nvfp4")
    oracle.store(rows[1], loc, v_ref, ps, "bf16", "nvfp4")
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    o_ref, l_ref = oracle.attention_rows(oracle.problem_for(w), w.q(), torch.from_numpy(k_ref),
                                         torch.from_numpy(v_ref), w.selected, w.block_tables, w.cu_seqlens_q,
                                         w.used_kv_lens)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, "store then attend")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, "store then attend lse")
