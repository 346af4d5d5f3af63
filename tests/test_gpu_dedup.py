"""GPU parity of the cross-sequence dedup path: mxsa_build_index_dedup, the
scheduler on its index and the forward on keys that hold rows of several
sequences, against the oracle (oracle.build_index_dedup, oracle.schedule,
oracle.attention_rows).

Index and schedule: bit-exact.  Output: the tolerances of the plain path
(dedup changes which key a row's block is computed under, not the result).
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


def _pair_edges():
    """64-token pages: sequence 1 shares both pages of blocks 0-2 with
    sequence 0; sequence 2 shares only the first page of block 0's pair (not
    shareable with 0); sequence 3 holds sequence 0's block-1 pages at its
    logical block 2 (another position: not shared) and sequence 0's block-0
    pages at block 0 (shared); sequence 4's block 3 is partial in it (never
    shared) though its pages equal sequence 0's."""
    w = W.custom("pair_edges", [1, 1, 2, 1, 3], [1000, 900, 800, 1100, 480], 16, 2, 64, 6, True, "uniform", 131)
    bt = w.block_tables
    bt[1, 0:6] = bt[0, 0:6]
    bt[2, 0] = bt[0, 0]
    bt[3, 4:6] = bt[0, 2:4]
    bt[3, 0:2] = bt[0, 0:2]
    bt[4, 6:8] = bt[0, 6:8]
    return w


def _causal_shared():
    """Prefill rows of two sequences meet in shared keys whose block is
    diagonal for both (L 1000 / 300 new tokens and L 1200 / 500): each row
    needs its own sequence's causal position."""
    w = W.custom("causal_shared", [300, 500, 4], [1000, 1200, 700], 16, 2, 128, 6, True, "zipf_diag", 132)
    bt = w.block_tables
    bt[1, 0:7] = bt[0, 0:7]
    bt[2, 0:5] = bt[0, 0:5]
    return w


CASES = {
    "shared_prefix_decode": W.custom("shared_prefix_decode", [1] * 24, [9000, 3000, 700, 20000, 129, 8192] * 4,
                                     16, 2, 64, 16, False, "hot_groups", 114, extra={"shared_prefix_blocks": 64}),
    "shared_prefix_prefill": W.custom("shared_prefix_prefill", [1, 3, 0, 5] * 6, [9000, 4000, 300, 12000] * 6,
                                      8, 1, 128, 8, True, "hot_groups", 115, extra={"shared_prefix_blocks": 64}),
    # 24 sequences: hot sequences s and s + 16 of each group share pages
    "shared_fp8_g32": W.custom("shared_fp8_g32", [1, 9, 1, 40] * 6, [5000, 2600, 7000, 3000] * 6, 32, 1, 64, 12,
                               True, "hot_groups", 133, kv_dtype="fp8", extra={"shared_prefix_blocks": 64}),
    "pair_edges": _pair_edges(),
    "causal_shared": _causal_shared(),
    # no page is shared: the dedup index equals the plain one
    "no_sharing": W.custom("no_sharing", [1, 8, 64, 130], [300, 1000, 2100, 2900], 32, 4, 128, 6, True,
                           "uniform_drop10", 103, kv_dtype="fp8"),
}


def run_dedup(w, num_ctas=0):
    import block_sparse_attention_builder_gb300 as mx
    inp = U.device_inputs(w)
    attn = mx.SparseAttention(U.problem(w), "cuda", num_ctas, dedup=True)
    out, lse = attn(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"])
    torch.cuda.synchronize()
    return attn, out, lse, inp


def oracle_dedup(w):
    prob = oracle.problem_for(w)
    return oracle.build_index_dedup(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens, w.block_tables)


@pytest.fixture(scope="module")
def runs():
    return {name: run_dedup(w) for name, w in CASES.items()}


@pytest.mark.parametrize("name", list(CASES))
def test_dedup_index_bit_exact(name, runs):
    w = CASES[name]
    got = U.read_index(runs[name][0])
    ref = oracle_dedup(w)
    assert got["nb"] == ref["nb"]
    assert got["flags"] == ref["flags"]
    for k in ("row_ptr", "entries", "slot_entry"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["active"], np.nonzero(np.diff(ref["row_ptr"]))[0])


@pytest.mark.parametrize("name", list(CASES))
def test_dedup_schedule_bit_exact(name, runs):
    w = CASES[name]
    prob = oracle.problem_for(w)
    ref = oracle.schedule(prob, w.used_kv_lens, w.cu_seqlens_q, oracle_dedup(w), U.ITEM_TILES, U.DECODE_BLOCKS,
                          NUM_SMS)
    got = U.read_sched(runs[name][0], NUM_SMS)
    for k in ("items", "cost_prefix", "cta_ptr", "items_dec", "cost_prefix_dec", "cta_ptr_dec"):
        assert np.array_equal(got[k], ref[k]), k


@pytest.mark.parametrize("name", list(CASES))
def test_dedup_end_to_end_matches_oracle(name, runs):
    w = CASES[name]
    attn, out, lse, _ = runs[name]
    assert attn.status() == 0
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, U.out_tol(w), f"{name} out")
    U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, f"{name} lse")


def test_sharing_merges_keys(runs):
    """Shared prefixes leave fewer active keys (blocks loaded) than the plain
    index, and a batch without shared pages leaves the plain index as is."""
    for name in ("shared_prefix_decode", "shared_prefix_prefill", "shared_fp8_g32", "causal_shared"):
        w = CASES[name]
        plain = oracle.build_index(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens)
        got = U.read_index(runs[name][0])
        assert got["n_active"] < np.count_nonzero(np.diff(plain["row_ptr"])), name
        assert got["nnz"] == len(plain["entries"]), name
    w = CASES["no_sharing"]
    plain = oracle.build_index(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens)
    got = U.read_index(runs["no_sharing"][0])
    for k in ("row_ptr", "entries", "slot_entry"):
        assert np.array_equal(got[k], plain[k]), k


def test_plan_after_dedup_restores_plain_rule(runs):
    """The plain plan on a workspace that last held a dedup index clears the
    dedup mark: the forward then takes causal positions per key again, and
    the output matches the oracle."""
    import block_sparse_attention_builder_gb300 as mx
    w = CASES["causal_shared"]
    attn, _, _, inp = runs["causal_shared"]
    mx.plan(attn.prob, inp["sel"], inp["cu"], inp["lens"], attn.ws.index, attn.ws.sched)
    out, lse = attn.attend(inp["q"], inp["k"], inp["v"], inp["bt"])
    torch.cuda.synchronize()
    L = mx.index_layout(attn.prob)
    assert int(attn.ws.index[L.header:L.header + 64].view(torch.int32)[10].item()) == 0
    o_ref, l_ref = U.oracle_full(w)
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, U.out_tol(w), "plain after dedup out")


@pytest.mark.parametrize("num_ctas", [1, 5])
def test_dedup_cta_count_does_not_change_result(num_ctas, runs):
    w = CASES["shared_prefix_prefill"]
    _, out0, lse0, _ = runs["shared_prefix_prefill"]
    _, out1, lse1, _ = run_dedup(w, num_ctas)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_dedup_full_size_skewed_decode():
    """The skewed decode batch with its hot groups' first 64 blocks on
    shared pages, at full size: index and schedule bit-exact, sampled rows
    against the oracle."""
    spec = W.WORKLOADS["skewed_decode"]
    w = W.make_workload(W.WorkloadSpec(**{**spec.__dict__, "extra": {**spec.extra, "shared_prefix_blocks": 64}}))
    attn, out, lse, _ = run_dedup(w)
    assert attn.status() == 0
    ref = oracle_dedup(w)
    got = U.read_index(attn)
    for k in ("row_ptr", "entries", "slot_entry"):
        assert np.array_equal(got[k], ref[k]), k
    prob = oracle.problem_for(w)
    ref_s = oracle.schedule(prob, w.used_kv_lens, w.cu_seqlens_q, ref, U.ITEM_TILES, U.DECODE_BLOCKS, NUM_SMS)
    got_s = U.read_sched(attn, NUM_SMS)
    for k in ("items", "cost_prefix", "cta_ptr", "items_dec", "cost_prefix_dec", "cta_ptr_dec"):
        assert np.array_equal(got_s[k], ref_s[k]), k
    rng = np.random.default_rng(1)
    G = w.num_q_heads // w.num_kv_heads
    pairs = np.unique(np.concatenate([[0, w.total_q * w.num_kv_heads - 1],
                                      rng.choice(w.total_q * w.num_kv_heads, size=24, replace=False)]))
    rows = (((pairs // w.num_kv_heads) * w.num_q_heads + (pairs % w.num_kv_heads) * G)[:, None]
            + np.arange(G)).reshape(-1)
    o_ref, l_ref = U.oracle_full(w, rows)
    o_gpu = out.float().reshape(-1, 128)[torch.from_numpy(rows).cuda()].cpu().numpy()
    l_gpu = lse.t().reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
    U.assert_close_out(o_gpu, o_ref, U.out_tol(w), "skewed dedup out")
    U.assert_close_lse(l_gpu, l_ref, 2e-3, "skewed dedup lse")
