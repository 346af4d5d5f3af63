"""Top-k block selection on the GPU (mxsa_select_blocks, through the C ABI)
against the oracle.  The selection is an integer decision, so both the block
scores (FP32, bit for bit, NaN where a block has no score) and the selected
blocks must be identical to the oracle's: small cases of both kernel forms
(one thread per key for sequences of at most 8 new tokens, one thread per
query for longer ones), index dims 64 and 128, every kv dtype, ties, NaN
keys, a bad cu_seqlens_q, sampled rows of two full-size workloads, and the
selections fed straight into the attention."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_attention_builder_gb300 as mx  # noqa: E402
import oracle  # noqa: E402
from block_sparse_attention_builder_gb300 import build as B  # noqa: E402
from block_sparse_attention_builder_gb300 import workloads as W  # noqa: E402
from tests import gpu_util as U  # noqa: E402

FLAG_CU = 128


def _w(name, tq, lens, hkv, ps, topk, causal, dtype, seed):
    return W.custom(name, tq, lens, hkv * 4, hkv, ps, topk, causal, "uniform", seed,
                    q_dtype="bf16" if dtype == "fp8" else dtype, kv_dtype=dtype)


def gpu_select(w, iq, ik, bt=None, cu=None):
    B.build()
    dev = "cuda"
    bt = torch.from_numpy(w.block_tables if bt is None else bt).to(dev)
    cu = torch.from_numpy(w.cu_seqlens_q if cu is None else cu).to(dev)
    lens = torch.from_numpy(w.used_kv_lens).to(dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    prob = U.problem(w)
    sel, ws = mx.select_blocks(prob, iq.to(dev), ik.to(dev), bt, cu, lens, flags=flags)
    torch.cuda.synchronize()
    nbm = (w.max_pages_per_seq * w.page_size + 127) // 128
    scores = ws[:w.total_q * w.num_kv_heads * nbm * 4].view(torch.float32).view(w.total_q, w.num_kv_heads, nbm)
    return sel.cpu().numpy(), scores.cpu().numpy(), int(flags.item())


def own_blocks(w, rows=None):
    """Mask [rows, nblk_max] of each row's own blocks (b < ceil(L / 128) of
    its sequence); the score workspace past them is unspecified."""
    nbm = (w.max_pages_per_seq * w.page_size + 127) // 128
    cap = w.max_pages_per_seq * w.page_size
    tok = np.arange(w.total_q) if rows is None else rows // w.num_kv_heads
    seq = np.searchsorted(w.cu_seqlens_q, tok, side="right") - 1
    L = np.clip(w.used_kv_lens[seq].astype(np.int64), 0, cap)
    return np.arange(nbm)[None, :] < ((L + 127) // 128)[:, None]


def assert_scores_equal(got, ref, what, mask=None):
    if mask is not None:
        got, ref = got[mask], ref[mask]
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: blocks with a score differ"
    assert np.array_equal(got[~nan_g].view(np.uint32), ref[~nan_r].view(np.uint32)), f"{what}: score bits differ"


CASES = [
    ("dec_fp8_64", [1, 1, 1], [300, 1000, 129], 2, 64, 4, False, "fp8", 11, 64),
    ("dec_bf16_128", [1, 1, 1, 1], [5000, 128, 777, 2048], 2, 64, 16, False, "bf16", 12, 128),
    ("short_fp16", [3, 8, 2], [700, 1300, 260], 2, 128, 6, True, "fp16", 13, 64),
    ("long_fp8", [200, 1, 37], [3000, 800, 1500], 2, 128, 12, True, "fp8", 14, 128),
    ("long_bf16_ps64", [130, 9], [2000, 1100], 1, 64, 20, True, "bf16", 15, 64),
    ("noncausal_long", [150], [4200], 2, 128, 40, False, "bf16", 16, 128),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_select_bit_exact_against_oracle(case):
    *spec, dim = case
    w = _w(*spec)
    iq, ik = w.idx_q(dim), w.idx_cache(dim)
    sel, scores, flags = gpu_select(w, iq, ik)
    ref_sel, ref_scores = oracle.select_blocks(oracle.problem_for(w), dim, iq, ik, w.block_tables, w.cu_seqlens_q,
                                               w.used_kv_lens, with_scores=True)
    assert flags == 0
    m = np.repeat(own_blocks(w)[:, None, :], w.num_kv_heads, axis=1)
    assert_scores_equal(scores, ref_scores, case[0], m)
    assert np.array_equal(sel, ref_sel), case[0]


def test_ties_nan_keys_and_padding():
    w = _w("ties", [1, 12], [1024, 640], 1, 128, 10, True, "fp8", 21)
    dim = 64
    iq, ik = w.idx_q(dim), w.idx_cache(dim).clone()
    bt = w.block_tables
    for dst in (5, 2):  # three equal blocks in sequence 0
        ik[int(bt[0, dst])] = ik[int(bt[0, 6])]
    ik.view(torch.uint8)[int(bt[1, 1])] = 0x7F  # a block of NaN keys in sequence 1
    sel, scores, _ = gpu_select(w, iq, ik)
    ref_sel, ref_scores = oracle.select_blocks(oracle.problem_for(w), dim, iq, ik, bt, w.cu_seqlens_q,
                                               w.used_kv_lens, with_scores=True)
    m = np.repeat(own_blocks(w)[:, None, :], w.num_kv_heads, axis=1)
    assert_scores_equal(scores, ref_scores, "ties", m)
    assert np.array_equal(sel, ref_sel)
    assert [b for b in sel[0, 0] if b in (2, 5, 6)] == [2, 5, 6]
    assert 1 not in sel[1:, 0]


def test_bad_cu_is_flagged_and_selects_nothing():
    w = _w("badcu", [2, 2], [300, 300], 1, 128, 3, False, "bf16", 22)
    cu = np.array([0, 3, 2], dtype=np.int64)
    sel, _, flags = gpu_select(w, w.idx_q(64), w.idx_cache(64), cu=cu)
    assert flags & FLAG_CU and (sel == -1).all()


def _sampled(name, dim, seqs):
    """A full-size workload: the GPU selects every row; the oracle checks
    the rows of a few sequences on a compact copy of their index pages."""
    w = W.workload(name)
    dev = "cuda"
    iq = w.idx_q(dim, dev)
    ik = w.idx_cache(dim, dev)
    sel, scores, flags = gpu_select(w, iq, ik)
    assert flags == 0
    # compact index cache: every page of the chosen sequences
    pages = sorted({int(p) for s in seqs for p in w.block_tables[s] if p >= 0})
    remap = {p: i for i, p in enumerate(pages)}
    bt = np.full_like(w.block_tables, -1)
    for s in seqs:
        for j, p in enumerate(w.block_tables[s]):
            if p >= 0:
                bt[s, j] = remap[int(p)]
    ikc = w.idx_cache_pages(dim, np.array(pages), dev)
    prob = oracle.problem_for(w)
    prob.num_pages = len(pages)
    rows = np.concatenate([np.arange(w.cu_seqlens_q[s] * w.num_kv_heads, w.cu_seqlens_q[s + 1] * w.num_kv_heads)
                           for s in seqs])
    if len(rows) > 96:
        rows = np.sort(np.random.default_rng(3).choice(rows, 96, replace=False))
    ref_sel, ref_scores = oracle.select_blocks(prob, dim, iq.cpu(), ikc, bt, w.cu_seqlens_q, w.used_kv_lens,
                                               with_scores=True, rows=rows)
    T, H = w.total_q, w.num_kv_heads
    t, g = rows // H, rows % H
    assert_scores_equal(scores[t, g], ref_scores[t, g], name, own_blocks(w, rows))
    assert np.array_equal(sel[t, g], ref_sel[t, g]), name


def test_full_size_gqa_decode_sampled_rows():
    _sampled("gqa_decode", 64, [0, 17, 33, 63])


def test_full_size_shared_prefill_sampled_rows():
    _sampled("shared_prefill", 128, [0])


def test_selections_feed_the_attention():
    """GPU selection, then the plan, forward and combine on those selections,
    against the oracle's attention over the oracle's own selections."""
    w = _w("e2e", [1, 40, 3], [900, 2600, 1500], 2, 64, 8, True, "bf16", 31)
    dim = 64
    iq, ik = w.idx_q(dim), w.idx_cache(dim)
    sel, _, _ = gpu_select(w, iq, ik)
    ref_sel = oracle.select_blocks(oracle.problem_for(w), dim, iq, ik, w.block_tables, w.cu_seqlens_q,
                                   w.used_kv_lens)
    assert np.array_equal(sel, ref_sel)
    w.selected = sel
    _, out, lse, _ = U.run(w)
    w.selected = ref_sel
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, U.out_tol(w), "e2e out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, "e2e lse")
