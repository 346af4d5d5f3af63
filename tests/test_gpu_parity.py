"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Index and schedule: bit-exact.  Forward partials and combine: checked in
isolation and end to end at fixed tolerances (BF16 / FP16 output
atol = rtol = 1e-2, FP8 4e-2, lse 2e-3 absolute).  The small
cases span several tiles per key and ragged tails; the full-size workloads
are checked bit-exactly for index and schedule and on sampled rows for the
output.
"""
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


def small_cases():
    return {
        "tiny_decode": W.workload("tiny_decode"),
        "gqa_decode_small": W.custom("gqa_decode_small", [1] * 6, [2100, 2500, 3333, 4096, 4097, 5000], 64, 8, 64,
                                     16, False, "uniform_last", 101),
        "prefill_small": W.custom("prefill_small", [384], [2432], 16, 1, 128, 8, True, "zipf_diag", 102),
        "fp8_varlen_small": W.custom("fp8_varlen_small", [1, 8, 64, 130], [300, 1000, 2100, 2900], 32, 4, 128, 6,
                                     True, "uniform_drop10", 103, kv_dtype="fp8"),
        "skewed_small": W.custom("skewed_small", [1] * 16, [200, 700, 1500, 9000] * 4, 64, 8, 64, 64, False,
                                 "hot_groups", 104),
        "fp16_gqa3": W.custom("fp16_gqa3", [2, 5, 1], [700, 1300, 129], 12, 4, 64, 5, True, "uniform", 105,
                              q_dtype="fp16", kv_dtype="fp16"),
        "mha_fp16_fp8": W.custom("mha_fp16_fp8", [3, 4], [640, 1111], 4, 4, 128, 4, True, "uniform", 106,
                                 q_dtype="fp16", kv_dtype="fp8"),
        "decode_edges": _decode_edge_workload(),
        # G = 32 and 64: the KV-stationary q boxes of an entry span one or
        # two warps' rows (decode rows go through the tile path too: G > 16)
        "g32_prefill": W.custom("g32_prefill", [1, 37, 90], [700, 1500, 2600], 32, 1, 128, 5, True, "zipf_diag",
                                110),
        "g64_mixed": W.custom("g64_mixed", [1, 3, 20], [200, 900, 1300], 64, 1, 64, 4, True, "uniform", 111,
                              q_dtype="fp16", kv_dtype="fp16"),
        # G = 128 (the largest): one entry per tile, a 128-row q box
        "g128_tiny": W.custom("g128_tiny", [1, 6], [300, 800], 128, 1, 64, 3, True, "uniform", 112),
        # top-k 256 (the largest): 256 slots per row through the index's
        # per-row ranking and the combine's slot loop
        "topk256": W.custom("topk256", [1, 50], [40000, 36000], 8, 1, 128, 256, True, "uniform", 113),
        # shared-prefix page tables: hot sequences s and s + 16 of a group
        # point their first 64 blocks at the same pages (the plain index
        # keeps one key per sequence; the pages are read once per sequence)
        "shared_prefix_decode": W.custom("shared_prefix_decode", [1] * 24, [9000, 3000, 700, 20000, 129, 8192] * 4,
                                         16, 2, 64, 16, False, "hot_groups", 114,
                                         extra={"shared_prefix_blocks": 64}),
        "shared_prefix_prefill": W.custom("shared_prefix_prefill", [1, 3, 0, 5] * 6, [9000, 4000, 300, 12000] * 6,
                                          8, 1, 128, 8, True, "hot_groups", 115,
                                          extra={"shared_prefix_blocks": 64}),
    }


def _decode_edge_workload():
    # An all-decode batch (every sequence has one new token or none), which
    # the plan indexes in its one-barrier form: seq 0 has a token but L = 0
    # (its selection is out of range, causal-length flag); seq 1 has no
    # token; seq 2's token selects nothing; seq 3 has an out-of-range and a
    # duplicate slot; seq 4 ends in a partial block; seq 5 is long.
    w = W.custom("decode_edges", [1, 0, 1, 1, 1, 1], [0, 300, 700, 1000, 333, 5000], 8, 2, 64, 6, True,
                 "uniform", 109)
    sel = w.selected
    sel[0] = -1
    sel[0, 1, 2] = 0          # L = 0: no block exists
    sel[1] = -1               # seq 2: nothing selected
    sel[2, 0, 1] = 99         # out of range
    sel[2, 1, 3] = sel[2, 1, 0]  # duplicate
    return w


SMALL = small_cases()


@pytest.fixture(scope="module")
def small_runs():
    return {name: U.run(w) for name, w in SMALL.items()}


@pytest.mark.parametrize("name", list(SMALL))
def test_index_bit_exact(name, small_runs):
    w = SMALL[name]
    attn = small_runs[name][0]
    got = U.read_index(attn)
    ref = oracle.build_index(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens)
    assert got["nb"] == ref["nb"]
    assert got["flags"] == ref["flags"]
    assert np.array_equal(got["row_ptr"], ref["row_ptr"])
    assert np.array_equal(got["entries"], ref["entries"])
    assert np.array_equal(got["slot_entry"], ref["slot_entry"])
    counts = np.diff(ref["row_ptr"])
    assert np.array_equal(got["active"], np.nonzero(counts)[0])


@pytest.mark.parametrize("name", list(SMALL))
def test_schedule_bit_exact(name, small_runs):
    w = SMALL[name]
    attn = small_runs[name][0]
    ref = U.oracle_schedule(w, NUM_SMS)
    got = U.read_sched(attn, NUM_SMS)
    assert got["num_ctas"] == NUM_SMS
    for k in ("items", "cost_prefix", "cta_ptr", "items_dec", "cost_prefix_dec", "cta_ptr_dec"):
        assert np.array_equal(got[k], ref[k]), k


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_partials_match_oracle(name, small_runs):
    """Partials straight out of the forward kernels.  Entries of normal items
    hold one block each; a decode item holds the merge of its run of blocks
    at its first entry (checked against the oracle's LSE merge of the run's
    per-block results) and -inf lse at the others."""
    w = SMALL[name]
    attn = small_runs[name][0]
    G = w.num_q_heads // w.num_kv_heads
    idx = U.read_index(attn)
    sch = U.read_sched(attn, NUM_SMS)
    o_gpu, l_gpu = U.read_partials(attn)
    o_ref, l_ref = U.oracle_slot_partials(w)
    # normal entries: one block per partial
    ents = np.concatenate([np.arange(e0, e0 + n) for _, e0, n, _ in sch["items"]]) if len(sch["items"]) else \
        np.zeros(0, np.int64)
    slots = idx["entries"][ents]
    rows_gpu = (ents[:, None] * G + np.arange(G)).reshape(-1)
    rows_ref = (slots[:, None] * G + np.arange(G)).reshape(-1)
    U.assert_close_out(o_gpu[rows_gpu], o_ref[rows_ref], U.out_tol(w), f"{name} partial o")
    U.assert_close_lse(l_gpu[rows_gpu], l_ref[rows_ref], 2e-3, f"{name} partial lse")
    # decode items: merged partial at the first entry, -inf elsewhere
    for a0, e0, _, nk in sch["items_dec"]:
        keys = idx["active"][a0:a0 + nk]
        es = idx["row_ptr"][keys]
        assert es[0] == e0
        sl = idx["entries"][es]
        for j in range(G):
            mo, ml = oracle.combine(o_ref[sl * G + j], l_ref[sl * G + j])
            U.assert_close_out(o_gpu[e0 * G + j], mo, U.out_tol(w), f"{name} decode partial o")
            U.assert_close_lse([l_gpu[e0 * G + j]], [ml], 2e-3, f"{name} decode partial lse")
            assert np.all(l_gpu[es[1:] * G + j] == -np.inf)


@pytest.mark.parametrize("name", list(SMALL))
def test_end_to_end_matches_oracle(name, small_runs):
    w = SMALL[name]
    _, out, lse, _ = small_runs[name]
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, U.out_tol(w), f"{name} out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, f"{name} lse")


def test_combine_with_oracle_partials():
    """The combine kernel alone, fed partials made by the oracle."""
    import block_sparse_attention_builder_gb300 as mx
    w = SMALL["fp16_gqa3"]
    attn, _, _, inp = U.run(w)
    G = w.num_q_heads // w.num_kv_heads
    idx = U.read_index(attn)
    o_ref, l_ref = U.oracle_slot_partials(w)
    nslots = len(idx["slot_entry"])
    o_buf = np.zeros((nslots * G, 128), np.float32)
    l_buf = np.full(nslots * G, -np.inf, np.float32)
    slots = np.nonzero(idx["slot_entry"] >= 0)[0]
    e = idx["slot_entry"][slots]
    for j in range(G):
        o_buf[e * G + j] = o_ref[slots * G + j]
        l_buf[e * G + j] = l_ref[slots * G + j]
    U.write_partials(attn, o_buf, l_buf)  # o rounded to the partial type, as the forward stores it
    out = torch.empty_like(inp["q"])
    lse = torch.empty(w.num_q_heads, w.total_q, dtype=torch.float32, device="cuda")
    mx.combine(attn.prob, attn.ws.index, attn.ws.partial, out, lse)
    torch.cuda.synchronize()
    full_o, full_l = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), full_o, 1e-2, "combine out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), full_l, 1e-5, "combine lse")


@pytest.mark.parametrize("name", ["fp8_varlen_small", "skewed_small", "edges", "decode_edges", "decode_bad_cu"])
def test_plan_equals_separate_index_and_schedule(name):
    """mxsa_plan (one launch) leaves the same index and schedule as
    mxsa_build_index followed by mxsa_schedule."""
    import block_sparse_attention_builder_gb300 as mx
    w = _edge_workload() if name == "edges" else SMALL["decode_edges" if name == "decode_bad_cu" else name]
    inp = U.device_inputs(w)
    if name == "decode_bad_cu":  # not a non-decreasing partition: nothing is indexed, CU flagged
        inp["cu"] = torch.tensor([0, 2, 1, 3, 4, 5, 5], dtype=torch.int64, device="cuda")
    prob = U.problem(w)
    a = mx.SparseAttention(prob, "cuda")
    b = mx.SparseAttention(prob, "cuda")
    mx.plan(prob, inp["sel"], inp["cu"], inp["lens"], a.ws.index, a.ws.sched)
    mx.build_index(prob, inp["sel"], inp["cu"], inp["lens"], b.ws.index)
    mx.schedule(prob, b.ws.index, b.ws.sched)
    torch.cuda.synchronize()
    ia, ib = U.read_index(a), U.read_index(b)
    for k in ia:
        assert np.array_equal(np.asarray(ia[k]), np.asarray(ib[k])), k
    sa, sb = U.read_sched(a, NUM_SMS), U.read_sched(b, NUM_SMS)
    for k in sa:
        assert np.array_equal(np.asarray(sa[k]), np.asarray(sb[k])), k
    if name == "decode_bad_cu":
        assert ia["flags"] & 128 and ia["nnz"] == 0
        assert np.all(ia["slot_entry"] == -1)
    if name == "decode_edges":
        assert ia["flags"] & 1 and ia["flags"] & 2 and ia["flags"] & 8


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_cta_count_does_not_change_result(num_ctas, small_runs):
    w = SMALL["prefill_small"]
    _, out0, lse0, inp = small_runs["prefill_small"]
    _, out1, lse1, _ = U.run(w, inp, num_ctas=num_ctas)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


@pytest.mark.parametrize("name", ["prefill_small", "fp8_varlen_small"])
def test_repeated_forward_on_one_plan(name):
    """The forward claims KV-stationary items from a counter in the schedule
    header; the last CTA to leave resets it, so forwards repeated on one plan
    see every item again and give bit-identical results."""
    import block_sparse_attention_builder_gb300 as mx
    w = SMALL[name]
    inp = U.device_inputs(w)
    attn = mx.SparseAttention(U.problem(w), "cuda")
    attn.prepare(inp["sel"], inp["cu"], inp["lens"])
    outs = [attn.attend(inp["q"], inp["k"], inp["v"], inp["bt"]) for _ in range(3)]
    torch.cuda.synchronize()
    assert attn.status() == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(outs[-1][0].float().cpu().numpy().reshape(-1, 128), o_ref, U.out_tol(w), f"{name} out")


def test_deterministic_repeat(small_runs):
    w = SMALL["skewed_small"]
    _, out0, lse0, inp = small_runs["skewed_small"]
    _, out1, lse1, _ = U.run(w, inp)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_softmax_scale():
    w = SMALL["gqa_decode_small"]
    _, out, lse, _ = U.run(w, scale=0.05)
    prob = oracle.problem_for(w, softmax_scale=0.05)
    o_ref, l_ref = oracle.attention_rows(prob, w.q(), w.k_cache(), w.v_cache(), w.selected, w.block_tables,
                                         w.cu_seqlens_q, w.used_kv_lens)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, "scale out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, "scale lse")


# ------------------------------------------------------- many sequences
def _many_seq_workload(name, tq, seed):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(130, 900, len(tq))]
    return W.custom(name, tq, lens, 8, 1, 64, 3, True, "uniform", seed)


@pytest.mark.parametrize("name,tq,seed", [
    # an all-decode batch past the 512 sequences of the plan's one-barrier
    # form: the general form indexes it
    ("decode_600", [1] * 600, 120),
    # past the 1024 sequences whose scan every CTA repeats: one CTA scans
    # and a grid barrier publishes the table
    ("mixed_1100", ([1, 1, 0, 2] * 275), 121),
])
def test_many_sequences(name, tq, seed):
    """Index and schedule bit-exact, the fused plan equal to the separate
    calls, and the output against the oracle, for batches of many
    sequences."""
    import block_sparse_attention_builder_gb300 as mx
    w = _many_seq_workload(name, tq, seed)
    attn, out, lse, inp = U.run(w)
    assert attn.status() == 0
    got = U.read_index(attn)
    ref = oracle.build_index(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens)
    assert got["flags"] == ref["flags"] == 0
    for k in ("row_ptr", "entries", "slot_entry"):
        assert np.array_equal(got[k], ref[k]), k
    sch, sref = U.read_sched(attn, NUM_SMS), U.oracle_schedule(w, NUM_SMS)
    for k in ("items", "cost_prefix", "cta_ptr", "items_dec", "cost_prefix_dec", "cta_ptr_dec"):
        assert np.array_equal(sch[k], sref[k]), k
    b = mx.SparseAttention(attn.prob, "cuda")
    mx.build_index(attn.prob, inp["sel"], inp["cu"], inp["lens"], b.ws.index)
    mx.schedule(attn.prob, b.ws.index, b.ws.sched)
    torch.cuda.synchronize()
    gb = U.read_index(b)
    for k in got:
        assert np.array_equal(np.asarray(got[k]), np.asarray(gb[k])), k
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, f"{name} out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, f"{name} lse")


# ------------------------------------------------------------------ edges
def _edge_workload():
    # seq 0: empty (L = 0, no tokens); seq 1: all slots -1 for token 0; seq 2:
    # a zero-token sequence between others; seq 3: out-of-range and duplicate
    # selections; every token of seq 4 selects its hot block 0
    w = W.custom("edges", [0, 2, 0, 3, 40], [0, 300, 128, 500, 4000], 8, 2, 64, 4, True, "uniform", 107)
    sel = w.selected
    sel[0] = -1                      # token 0 (seq 1): nothing selected
    sel[2, 0, 1] = 99                # out of range
    sel[3, 1, 2] = sel[3, 1, 0]      # duplicate
    for t in range(5, 45):
        sel[t, :, 0] = 0
        for g in range(2):
            row = sel[t, g]
            dup = [k for k in range(1, 4) if row[k] == 0]
            for k in dup:
                row[k] = -1
    return w


def test_edge_cases_match_oracle_and_flags():
    w = _edge_workload()
    attn, out, lse, _ = U.run(w)
    flags = attn.status()
    ref_idx = oracle.build_index(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens)
    assert flags == ref_idx["flags"] and flags & 1 and flags & 2
    got = U.read_index(attn)
    assert np.array_equal(got["entries"], ref_idx["entries"])
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, "edges out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, "edges lse")
    assert torch.all(out[0] == 0) and torch.all(torch.isinf(lse[:, 0]))


def test_quickstart_call_shape():
    import block_sparse_attention_builder_gb300 as mx
    w = W.custom("quick", [1], [256], 16, 1, 64, 2, False, "all", 108)
    inp = U.device_inputs(w)
    out, lse = mx.kvouter_attention(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"],
                                    page_size=64, return_lse=True)
    assert out.shape == (1, 16, 128) and out.dtype == torch.bfloat16
    assert lse.shape == (16, 1) and lse.dtype == torch.float32
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, 1e-2, "quickstart")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, "quickstart lse")


def test_pinned_host_outputs_and_pageable_refused():
    """out / lse in pinned host memory are written by the combine kernel
    directly (same values as device outputs); pageable host memory is refused
    by the binding and by the library before any launch."""
    import block_sparse_attention_builder_gb300 as mx
    w = SMALL["gqa_decode_small"]
    inp = U.device_inputs(w)
    attn = mx.SparseAttention(U.problem(w), "cuda")
    out_d, lse_d = attn(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"])
    h_out = torch.full(out_d.shape, 7.0, dtype=out_d.dtype).pin_memory()
    h_lse = torch.full(lse_d.shape, 7.0, dtype=torch.float32).pin_memory()
    attn.prepare(inp["sel"], inp["cu"], inp["lens"])
    attn.attend(inp["q"], inp["k"], inp["v"], inp["bt"], out=h_out, lse=h_lse)
    torch.cuda.synchronize()
    assert torch.equal(h_out, out_d.cpu()) and torch.equal(h_lse, lse_d.cpu())
    pageable = torch.empty(out_d.shape, dtype=out_d.dtype)
    with pytest.raises(ValueError):
        attn.attend(inp["q"], inp["k"], inp["v"], inp["bt"], out=pageable)
    with pytest.raises(mx.MxsaError) as ei:
        mx.combine(attn.prob, attn.ws.index, attn.ws.partial, pageable)
    assert ei.value.status == 1


def test_bad_page_id_is_flagged_not_faulted():
    import block_sparse_attention_builder_gb300 as mx
    w = W.workload("tiny_decode")
    inp = U.device_inputs(w)
    b = w.block_tables.copy()
    b[0, 0] = 10 ** 6
    inp["bt"] = torch.from_numpy(b).cuda()
    with pytest.raises(mx.MxsaError) as ei:
        mx.kvouter_attention(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"],
                             page_size=64)
    assert ei.value.flags & 4


# ------------------------------------------------------- full-size workloads
FULL = ["gqa_decode", "shared_prefill", "fp8_varlen", "skewed_decode"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    w = W.workload(name)
    attn, out, lse, inp = U.run(w)
    assert attn.status() == 0
    prob = oracle.problem_for(w)
    # index and schedule: bit-exact
    ref_idx = oracle.build_index(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens)
    got = U.read_index(attn)
    assert np.array_equal(got["row_ptr"], ref_idx["row_ptr"])
    assert np.array_equal(got["entries"], ref_idx["entries"])
    assert np.array_equal(got["slot_entry"], ref_idx["slot_entry"])
    ref_s = U.oracle_schedule(w, NUM_SMS)
    got_s = U.read_sched(attn, NUM_SMS)
    for k in ("items", "cost_prefix", "cta_ptr", "items_dec", "cost_prefix_dec", "cta_ptr_dec"):
        assert np.array_equal(got_s[k], ref_s[k]), k
    # output on sampled rows: every head of ~2048 / (topk * 2) sampled
    # (token, kv head) pairs, always including the first and the last token
    rng = np.random.default_rng(0)
    G = w.num_q_heads // w.num_kv_heads
    n_pairs = max(4, 2048 // (w.topk * 2))
    pairs = rng.choice(w.total_q * w.num_kv_heads, size=min(n_pairs, w.total_q * w.num_kv_heads), replace=False)
    pairs = np.unique(np.concatenate([[0, w.total_q * w.num_kv_heads - 1], pairs]))
    rows = ((pairs // w.num_kv_heads) * w.num_q_heads + (pairs % w.num_kv_heads) * G)[:, None] + np.arange(G)
    rows = rows.reshape(-1)
    o_ref, l_ref = U.oracle_full(w, rows)
    o_gpu = out.float().reshape(-1, 128)[torch.from_numpy(rows).cuda()].cpu().numpy()
    l_gpu = lse.t().reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    U.assert_close_out(o_gpu, o_ref, U.out_tol(w), f"{name} out")
    U.assert_close_lse(l_gpu, l_ref, 2e-3, f"{name} lse")
    # properties at any size: finite output, lse finite where anything was selected
    assert torch.isfinite(out.float()).all()
