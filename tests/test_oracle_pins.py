"""Pins for the CPU oracle: each test checks it against something other than
itself -- torch's dense SDPA on contiguous K/V, SDPA with a mask built from
the selections, closed forms, invariances, torch's dtype conversions and a
brute-force per-key scan for the index.  A dropped term, a wrong sign, a
wrong page or head index, a wrong causal offset or a transposed operand in
the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_builder_gb300 import workloads as W
from tests.paged import contiguous_kv, scatter_pages

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- helpers
def _dense_reference(q, k_list, v_list, cu, lens, hq, hkv, causal, allowed=None, scale=None):
    """Reference out/lse per (t, h) with torch SDPA in float64.

    allowed: optional callable (t, g, L) -> bool mask [L] of keys the row may use.
    """
    G = hq // hkv
    D = 128
    scale = scale or 1.0 / math.sqrt(D)
    Tq = q.shape[0]
    out = torch.zeros(Tq, hq, D, dtype=torch.float64)
    lse = torch.full((Tq, hq), -math.inf, dtype=torch.float64)
    for s in range(len(lens)):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        L = int(lens[s])
        if t1 == t0 or L == 0:
            continue
        n = t1 - t0
        qs = q[t0:t1].to(torch.float64).permute(1, 0, 2)                  # [Hq, n, D]
        ks = k_list[s].to(torch.float64).repeat_interleave(G, dim=0)      # [Hq, L, D]
        vs = v_list[s].to(torch.float64).repeat_interleave(G, dim=0)
        mask = torch.ones(hq, n, L, dtype=torch.bool)
        if causal:
            i = torch.arange(n).view(n, 1)
            p = torch.arange(L).view(1, L)
            mask &= (p <= (L - n + i)).unsqueeze(0)
        if allowed is not None:
            for i in range(n):
                for h in range(hq):
                    mask[h, i] &= allowed(t0 + i, h // G, L)
        o = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=scale)
        sc = torch.matmul(qs, ks.transpose(1, 2)) * scale
        sc = sc.masked_fill(~mask, -math.inf)
        ls = torch.logsumexp(sc, dim=-1)                                   # [Hq, n]
        empty = ~mask.any(dim=-1)
        o = torch.where(empty.unsqueeze(-1), torch.zeros_like(o), o)
        out[t0:t1] = o.permute(1, 0, 2)
        lse[t0:t1] = ls.permute(1, 0)
    return out, lse


def _run_oracle(q, kc, vc, sel, bt, cu, lens, hq, hkv, ps, causal, q_dtype, kv_dtype, topk, scale=0.0):
    prob = oracle.problem(len(lens), q.shape[0], hq, hkv, topk, ps, kc.shape[0], bt.shape[1], causal,
                          q_dtype, kv_dtype, scale)
    out, lse = oracle.attention_rows(prob, q, kc, vc, sel, bt, cu, lens)
    return out.reshape(q.shape[0], hq, 128), lse.reshape(q.shape[0], hq)


def _case(seed, lens, tq, hq, hkv, ps, q_dtype="bf16", kv_dtype="bf16"):
    rng = np.random.default_rng(seed)
    k_list = contiguous_kv(seed, lens, hkv, kv_dtype, 2)
    v_list = contiguous_kv(seed, lens, hkv, kv_dtype, 3)
    kc, bt = scatter_pages(k_list, ps, np.random.default_rng(seed + 1))
    vc = torch.zeros_like(kc)
    # V pages go to the same physical pages as K (one block table)
    for s, x in enumerate(v_list):
        L = x.shape[1]
        for lp in range((L + ps - 1) // ps):
            n = min(ps, L - lp * ps)
            vc[bt[s, lp], :, :n, :] = x[:, lp * ps: lp * ps + n, :]
    total_q = int(sum(tq))
    q = W.generate_values(total_q * hq * 128, W.stream_key(seed, 1), q_dtype, "cpu").view(total_q, hq, 128)
    cu = np.zeros(len(tq) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(tq)
    return rng, q, k_list, v_list, kc, vc, bt, cu, np.asarray(lens, dtype=np.int32)


# ------------------------------------------------------------ dtype pins
def test_decode_bf16_all_codes():
    codes = np.arange(65536, dtype=np.uint32)
    ref = torch.from_numpy(codes.astype(np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode("bf16", c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_decode_fp16_all_codes():
    codes = np.arange(65536, dtype=np.uint32)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.decode("fp16", c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_decode_fp8_e4m3_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.decode("fp8", int(c)) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    assert np.nanmax(np.abs(got)) == 448.0


def test_fp8_input_cast_rule():
    # the generator's FP8 values follow x.float().clamp(-448, 448).to(float8_e4m3fn)
    t = W._quantile_table("fp8")
    from scipy.special import ndtri
    z = torch.from_numpy(ndtri((np.arange(65536) + 0.5) / 65536).astype(np.float32))
    ref = z.float().clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(t, ref)


# ------------------------------------------------- attention value pins
DENSE_CASES = [
    # lens, tq, hq, hkv, ps, causal, q_dtype, kv_dtype
    ([256], [1], 16, 1, 64, False, "bf16", "bf16"),
    ([300, 129, 1], [3, 2, 1], 8, 2, 64, True, "bf16", "bf16"),
    ([200, 385], [4, 1], 4, 4, 128, False, "fp16", "fp16"),
    ([513, 140], [5, 140], 16, 1, 128, True, "bf16", "fp8"),
    ([70], [2], 2, 1, 64, True, "bf16", "bf16"),
]


@pytest.mark.parametrize("case", DENSE_CASES)
def test_all_blocks_selected_equals_dense_sdpa(case):
    lens, tq, hq, hkv, ps, causal, qd, kd = case
    rng, q, k_list, v_list, kc, vc, bt, cu, lens_a = _case(7, lens, tq, hq, hkv, ps, qd, kd)
    nblk = [(L + 127) // 128 for L in lens]
    topk = max(nblk)
    sel = np.full((q.shape[0], hkv, topk), -1, dtype=np.int32)
    for s in range(len(lens)):
        for t in range(int(cu[s]), int(cu[s + 1])):
            for g in range(hkv):
                sel[t, g, :nblk[s]] = rng.permutation(nblk[s])
    out, lse = _run_oracle(q, kc, vc, sel, bt, cu, lens_a, hq, hkv, ps, causal, qd, kd, topk)
    ref_o, ref_l = _dense_reference(q, k_list, v_list, cu, lens_a, hq, hkv, causal)
    assert np.allclose(out, ref_o.numpy(), atol=1e-12, rtol=1e-10)
    assert np.allclose(lse, ref_l.numpy(), atol=1e-10, rtol=0)


SPARSE_CASES = [
    ([1000, 333, 640], [2, 3, 1], 8, 2, 64, False, 3),
    ([900, 1100], [6, 4], 16, 2, 128, True, 4),
    ([257], [257], 4, 1, 64, True, 2),
]


@pytest.mark.parametrize("case", SPARSE_CASES)
def test_sparse_selection_equals_masked_sdpa(case):
    lens, tq, hq, hkv, ps, causal, topk = case
    rng, q, k_list, v_list, kc, vc, bt, cu, lens_a = _case(11, lens, tq, hq, hkv, ps)
    sel = np.full((q.shape[0], hkv, topk), -1, dtype=np.int32)
    for s in range(len(lens)):
        nblk = (lens[s] + 127) // 128
        for t in range(int(cu[s]), int(cu[s + 1])):
            for g in range(hkv):
                n = int(rng.integers(0, min(topk, nblk) + 1))
                sel[t, g, :n] = rng.choice(nblk, n, replace=False)
                sel[t, g] = sel[t, g, rng.permutation(topk)]

    def allowed(t, g, L):
        blocks = set(int(b) for b in sel[t, g] if b >= 0)
        p = torch.arange(L)
        return torch.tensor([int(x) // 128 in blocks for x in p.tolist()], dtype=torch.bool)

    out, lse = _run_oracle(q, kc, vc, sel, bt, cu, lens_a, hq, hkv, ps, causal, "bf16", "bf16", topk)
    ref_o, ref_l = _dense_reference(q, k_list, v_list, cu, lens_a, hq, hkv, causal, allowed=allowed)
    assert np.allclose(out, ref_o.numpy(), atol=1e-12, rtol=1e-10)
    fin = np.isfinite(ref_l.numpy())
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(lse[fin], ref_l.numpy()[fin], atol=1e-10, rtol=0)
    assert np.all(lse[~fin] == -np.inf) and np.all(out[~fin] == 0)


def test_slot_permutation_invariance():
    w = W.custom("perm", [3, 2], [700, 1200], 8, 2, 64, 5, True, "uniform", 21)
    prob = oracle.problem_for(w)
    q, kc, vc = w.q(), w.k_cache(), w.v_cache()
    o1, l1 = oracle.attention_rows(prob, q, kc, vc, w.selected, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    rng = np.random.default_rng(3)
    sel2 = w.selected.copy()
    for t in range(sel2.shape[0]):
        for g in range(sel2.shape[1]):
            sel2[t, g] = sel2[t, g, rng.permutation(sel2.shape[2])]
    o2, l2 = oracle.attention_rows(prob, q, kc, vc, sel2, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_single_key_closed_form():
    # L = 1: the only key is position 0 -> out = v_0 exactly, lse = score
    rng, q, k_list, v_list, kc, vc, bt, cu, lens = _case(5, [1], [1], 4, 2, 64)
    sel = np.array([[[0], [0]]], dtype=np.int32)
    out, lse = _run_oracle(q, kc, vc, sel, bt, cu, lens, 4, 2, 64, False, "bf16", "bf16", 1)
    for h in range(4):
        g = h // 2
        v0 = v_list[0][g, 0].to(torch.float64).numpy()
        k0 = k_list[0][g, 0].to(torch.float64).numpy()
        q0 = q[0, h].to(torch.float64).numpy()
        assert np.array_equal(out[0, h], v0)
        assert abs(lse[0, h] - float(np.dot(q0, k0)) / math.sqrt(128)) < 1e-12


def test_causal_first_token_sees_one_key():
    # Tq = L (whole sequence is new): token 0 sits at position 0 and sees key 0 only
    rng, q, k_list, v_list, kc, vc, bt, cu, lens = _case(6, [130], [130], 2, 1, 64)
    sel = np.array([[[0, 1]]] * 130, dtype=np.int32)
    out, lse = _run_oracle(q, kc, vc, sel, bt, cu, lens, 2, 1, 64, True, "bf16", "bf16", 2)
    for h in range(2):
        assert np.array_equal(out[0, h], v_list[0][0, 0].to(torch.float64).numpy())
        s0 = float(np.dot(q[0, h].double().numpy(), k_list[0][0, 0].double().numpy())) / math.sqrt(128)
        assert abs(lse[0, h] - s0) < 1e-12


def test_softmax_scale_argument():
    rng, q, k_list, v_list, kc, vc, bt, cu, lens = _case(8, [300], [2], 4, 1, 128)
    sel = np.array([[[0, 1, 2]]] * 2, dtype=np.int32)
    out, lse = _run_oracle(q, kc, vc, sel, bt, cu, lens, 4, 1, 128, False, "bf16", "bf16", 3, scale=0.05)
    ref_o, ref_l = _dense_reference(q, k_list, v_list, cu, lens, 4, 1, False, scale=0.05)
    assert np.allclose(out, ref_o.numpy(), atol=1e-12) and np.allclose(lse, ref_l.numpy(), atol=1e-10)


def test_rows_are_convex_combinations_of_selected_values():
    w = W.custom("cvx", [2, 1], [900, 400], 8, 2, 128, 3, False, "uniform", 4)
    prob = oracle.problem_for(w)
    q, kc, vc = w.q(), w.k_cache(), w.v_cache()
    out, lse = oracle.attention_rows(prob, q, kc, vc, w.selected, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    vals = vc.to(torch.float64).numpy()
    G = 4
    for r in range(out.shape[0]):
        t, h = divmod(r, 8)
        s = int(np.searchsorted(w.cu_seqlens_q, t, side="right") - 1)
        L = int(w.used_kv_lens[s])
        vs = []
        for b in w.selected[t, h // G]:
            for p in range(128 * b, min(128 * b + 128, L)):
                vs.append(vals[w.block_tables[s, p // 128], h // G, p % 128])
        vs = np.array(vs)
        assert np.all(out[r] >= vs.min(0) - 1e-12) and np.all(out[r] <= vs.max(0) + 1e-12)


def test_empty_rows_and_zero_length_sequence():
    rng, q, k_list, v_list, kc, vc, bt, cu, lens = _case(9, [256, 1], [1, 1], 4, 1, 64)
    lens = np.array([256, 0], dtype=np.int32)
    sel = np.array([[[-1, -1]], [[0, -1]]], dtype=np.int32)  # row 0 selects nothing; seq 1 has no keys
    out, lse = _run_oracle(q, kc, vc, sel, bt, cu, lens, 4, 1, 64, False, "bf16", "bf16", 2)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_out_of_range_and_duplicate_selections():
    w = W.custom("dup", [2], [600], 4, 1, 64, 4, False, "uniform", 12)
    prob = oracle.problem_for(w)
    q, kc, vc = w.q(), w.k_cache(), w.v_cache()
    base = w.selected.copy()
    o1, l1 = oracle.attention_rows(prob, q, kc, vc, base, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    bad = base.copy()
    bad[0, 0, 1] = 99          # beyond nblk = 5: ignored
    bad[1, 0, 2] = bad[1, 0, 0]  # repeated block: set semantics
    ref = base.copy()
    ref[0, 0, 1] = -1
    ref[1, 0, 2] = -1
    o2, l2 = oracle.attention_rows(prob, q, kc, vc, bad, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    o3, l3 = oracle.attention_rows(prob, q, kc, vc, ref, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    assert np.array_equal(o2, o3) and np.array_equal(l2, l3)
    assert not np.array_equal(o1, o3)


# ------------------------------------------------------------ combine pins
def test_combine_of_block_partials_equals_single_softmax():
    w = W.custom("cmb", [3, 2], [1500, 900], 8, 2, 64, 6, True, "uniform", 13)
    prob = oracle.problem_for(w)
    q, kc, vc = w.q(), w.k_cache(), w.v_cache()
    full_o, full_l = oracle.attention_rows(prob, q, kc, vc, w.selected, w.block_tables, w.cu_seqlens_q,
                                           w.used_kv_lens)
    rng = np.random.default_rng(0)
    groups = rng.integers(0, 3, size=w.topk)  # a random partition of the slots into 3 groups
    parts_o, parts_l = [], []
    for grp in range(3):
        sel = w.selected.copy()
        sel[:, :, groups != grp] = -1
        o, l = oracle.attention_rows(prob, q, kc, vc, sel, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
        parts_o.append(o)
        parts_l.append(l)
    for r in range(full_o.shape[0]):
        o, l = oracle.combine(np.stack([p[r] for p in parts_o]), np.array([p[r] for p in parts_l]))
        assert np.allclose(o, full_o[r], atol=1e-12, rtol=1e-10)
        assert abs(l - full_l[r]) < 1e-10 or (l == full_l[r] == -np.inf)


def test_combine_closed_forms():
    o = np.arange(256, dtype=np.float64).reshape(2, 128)
    # equal weights: plain average, lse = lse0 + ln 2
    out, l = oracle.combine(o, np.array([1.5, 1.5]))
    assert np.allclose(out, o.mean(0)) and abs(l - (1.5 + math.log(2))) < 1e-15
    # an empty part carries no weight
    out, l = oracle.combine(o, np.array([0.25, -np.inf]))
    assert np.array_equal(out, o[0]) and l == 0.25
    out, l = oracle.combine(o, np.array([-np.inf, -np.inf]))
    assert np.all(out == 0) and l == -np.inf


# -------------------------------------------------------------- quick start
def test_quickstart_shapes_and_dense_equivalence():
    with open(os.path.join(GOLDEN, "quickstart.json")) as f:
        g = json.load(f)
    hq, hkv, ps = g["num_q_heads"], g["num_kv_heads"], g["page_size"]
    L = g["used_kv_lens"][0]
    rng, q, k_list, v_list, kc, vc, bt, cu, lens = _case(31, [L], [1], hq, hkv, ps)
    bt = np.array(g["block_tables"], dtype=np.int32)
    kc = torch.cat([k_list[0][:, i * ps:(i + 1) * ps].unsqueeze(0) for i in range(4)])
    vc = torch.cat([v_list[0][:, i * ps:(i + 1) * ps].unsqueeze(0) for i in range(4)])
    assert list(kc.shape) == g["k_cache_shape"]
    sel = np.array(g["selected"], dtype=np.int32)
    out, lse = _run_oracle(q, kc, vc, sel, bt, np.array(g["cu_seqlens_q"]), np.array(g["used_kv_lens"], np.int32),
                           hq, hkv, ps, False, "bf16", "bf16", sel.shape[2])
    assert list(out.shape) == g["output_shape"]
    assert list(lse.T.shape) == g["lse_shape"]
    ref_o, ref_l = _dense_reference(q, k_list, v_list, np.array(g["cu_seqlens_q"]), [L], hq, hkv, False)
    assert np.allclose(out, ref_o.numpy(), atol=1e-12) and np.allclose(lse, ref_l.numpy(), atol=1e-10)


# ---------------------------------------------------------------- index pins
def _brute_force_index(sel, cu, lens, hkv, causal, cap_len):
    """Per-key scan over all slots in slot order (O(keys * slots))."""
    B = len(lens)
    Lc = [min(max(int(L), 0), cap_len) for L in lens]
    nblk = [(L + 127) // 128 for L in Lc]
    topk = sel.shape[2]
    seq_of = {}
    for s in range(B):
        for t in range(int(cu[s]), int(cu[s + 1])):
            seq_of[t] = s
    row_ptr = [0]
    entries = []
    for g in range(hkv):
        for s in range(B):
            n = int(cu[s + 1] - cu[s])
            for b in range(nblk[s]):
                for t in range(int(cu[s]), int(cu[s + 1])):
                    pos = Lc[s] - n + (t - int(cu[s]))
                    row = list(sel[t, g])
                    if b in row and not (causal and 128 * b > pos):
                        k = row.index(b)  # first slot holding b
                        entries.append((t * hkv + g) * topk + k)
                row_ptr.append(len(entries))
    return np.array(row_ptr, np.int32), np.array(entries, np.int32)


@pytest.mark.parametrize("causal", [False, True])
def test_index_matches_brute_force_scan(causal):
    rng = np.random.default_rng(5 + causal)
    lens = np.array([700, 129, 0, 1300], dtype=np.int32)
    tq = [3, 1, 0, 5]
    hkv, topk = 2, 4
    cu = np.zeros(5, np.int64)
    cu[1:] = np.cumsum(tq)
    T = int(cu[-1])
    sel = np.full((T, hkv, topk), -1, np.int32)
    for s in range(4):
        nb = (lens[s] + 127) // 128
        for t in range(int(cu[s]), int(cu[s + 1])):
            for g in range(hkv):
                n = min(topk, nb)
                sel[t, g, :n] = rng.choice(nb, n, replace=False)
                sel[t, g] = sel[t, g, rng.permutation(topk)]
    sel[0, 0, 0] = 50           # out of range
    sel[4, 1, 3] = sel[4, 1, 1]  # duplicate (keep the first)
    prob = oracle.problem(4, T, 8, hkv, topk, 64, 100, 21, causal)
    idx = oracle.build_index(prob, sel, cu, lens)
    rp, ent = _brute_force_index(np.where(sel == 50, -1, sel), cu, lens, hkv, causal, 21 * 64)
    assert np.array_equal(idx["row_ptr"], rp)
    assert np.array_equal(idx["entries"], ent)
    assert idx["flags"] & 1 and idx["flags"] & 2
    # slot_entry is the inverse permutation of entries
    se = idx["slot_entry"]
    assert np.array_equal(se[ent], np.arange(len(ent)))
    assert (se >= 0).sum() == len(ent)


def test_index_invalid_cu_indexes_nothing():
    sel = np.zeros((3, 1, 1), np.int32)
    prob = oracle.problem(2, 3, 1, 1, 1, 64, 4, 4, False)
    idx = oracle.build_index(prob, sel, np.array([0, 2, 1], np.int64), np.array([200, 200], np.int32))
    assert idx["flags"] & 128 and len(idx["entries"]) == 0 and np.all(idx["slot_entry"] == -1)


def test_index_flags_len_and_causal():
    sel = np.zeros((2, 1, 1), np.int32)
    cu = np.array([0, 2], np.int64)
    prob = oracle.problem(1, 2, 1, 1, 1, 64, 4, 2, True)
    idx = oracle.build_index(prob, sel, cu, np.array([1], np.int32))  # L < Tq with causal
    assert idx["flags"] & 8
    idx = oracle.build_index(prob, sel, cu, np.array([500], np.int32))  # L beyond 2 pages * 64
    assert idx["flags"] & 16


# ------------------------------------------------------------- schedule pins
def test_schedule_split_worked_example():
    # one key with 10 entries (a 10-token sequence: normal list), G = 32 ->
    # 4 entries per tile, 1 tile per item: n = ceil(10 / 4) = 3 items with
    # boundaries floor(i*10/3) = 0, 3, 6, 10
    sel = np.zeros((10, 1, 1), np.int32)
    cu = np.array([0, 10], np.int64)
    prob = oracle.problem(1, 10, 32, 1, 1, 128, 1, 1, False)
    idx = oracle.build_index(prob, sel, cu, np.array([100], np.int32))
    sch = oracle.schedule(prob, [100], cu, idx, 1, 16, 2)
    assert sch["items"][:, 1].tolist() == [0, 3, 6] and sch["items"][:, 2].tolist() == [3, 3, 4]
    # cost = 384 per item + 100 tokens * 2 + 1 tile * 256 + rows * 3, rows =
    # entries * 32: 384 + 200 + 256 + 288 = 1128 (3 entries) and
    # 384 + 200 + 256 + 384 = 1224 (4 entries)
    assert sch["cost_prefix"].tolist() == [0, 1128, 2256, 3480]
    # targets floor(c * 3480 / 2) = 0, 1740, 3480 -> items with prefix below them
    assert sch["cta_ptr"].tolist() == [0, 2, 3]
    assert len(sch["items_dec"]) == 0 and sch["cta_ptr_dec"].tolist() == [0, 0, 0]


def test_schedule_decode_run_worked_example():
    # one decode token (Tq = 1), G = 8, selecting 20 of the 25 blocks of a
    # 3100-token sequence: one run of 20 keys -> ceil(20 / 16) = 2 items of
    # run positions [0, 10) and [10, 20); the last block (24) holds 3100 - 3072
    # = 28 tokens.  cost = sum valid * 2 + 10 * 64 + 256
    blocks = np.array([24, 0, 3, 5, 7, 9, 11, 13, 15, 17, 19, 21, 23, 1, 2, 4, 6, 8, 10, 12], np.int32)
    sel = blocks.reshape(1, 1, 20)
    cu = np.array([0, 1], np.int64)
    prob = oracle.problem(1, 1, 8, 1, 20, 64, 49, 49, False)
    idx = oracle.build_index(prob, sel, cu, np.array([3100], np.int32))
    sch = oracle.schedule(prob, [3100], cu, idx, 4, 16, 3)
    assert len(sch["items"]) == 0
    d = sch["items_dec"]
    assert d[:, 0].tolist() == [0, 10] and d[:, 3].tolist() == [10, 10] and d[:, 2].tolist() == [1, 1]
    # entries follow key order (block order): the first key of item 1 is the
    # 11th smallest selected block
    assert d[:, 1].tolist() == [0, 10]
    first = 10 * 128 * 2 + 10 * 64 + 256
    second = (9 * 128 + 28) * 2 + 10 * 64 + 256
    assert sch["cost_prefix_dec"].tolist() == [0, first, first + second]


def test_schedule_decode_run_of_a_multiple_of_the_item_size():
    # a run of 16 keys with 8 keys per decode item: exactly 2 items of 8
    sel = np.arange(16, dtype=np.int32).reshape(1, 1, 16)
    cu = np.array([0, 1], np.int64)
    prob = oracle.problem(1, 1, 8, 1, 16, 64, 32, 32, False)
    idx = oracle.build_index(prob, sel, cu, np.array([2048], np.int32))
    sch = oracle.schedule(prob, [2048], cu, idx, 4, 8, 2)
    assert sch["items_dec"][:, 0].tolist() == [0, 8] and sch["items_dec"][:, 3].tolist() == [8, 8]


@pytest.mark.parametrize("name", ["tiny_decode", "shared_prefill_small", "varlen_small", "skewed_small"])
def test_schedule_invariants(name):
    if name == "shared_prefill_small":
        w = W.custom(name, [256], [2048], 16, 1, 128, 8, True, "zipf_diag", 3)
    elif name == "varlen_small":
        w = W.custom(name, [1, 8, 64, 3, 1], [3000, 900, 2000, 5000, 700], 32, 4, 128, 6, True, "uniform_drop10", 4)
    elif name == "skewed_small":
        w = W.custom(name, [1] * 16, [200, 700, 1500, 9000] * 4, 64, 8, 64, 64, False, "hot_groups", 104)
    else:
        w = W.workload(name)
    prob = oracle.problem_for(w)
    idx = oracle.build_index(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens)
    G = w.num_q_heads // w.num_kv_heads
    rp = idx["row_ptr"]
    active = np.nonzero(np.diff(rp))[0]
    tq = np.diff(w.cu_seqlens_q)
    for R, D in ((1, 16), (4, 8)):
        for P in (1, 7, 152):
            sch = oracle.schedule(prob, w.used_kv_lens, w.cu_seqlens_q, idx, R, D, P)
            covered = []
            for key, e0, n, _ in sch["items"]:
                assert rp[key] <= e0 and e0 + n <= rp[key + 1]
                assert 1 <= n <= R * max(1, 128 // G)
                covered.extend(range(e0, e0 + n))
            for a0, e, one, nk in sch["items_dec"]:
                assert one == 1 and 1 <= nk <= D and e == rp[active[a0]]
                keys = active[a0:a0 + nk]
                assert np.all(np.diff(rp)[keys] == 1)  # one entry per decode key
                covered.extend(rp[keys].tolist())
                # a decode item stays within one (kv head, sequence): same token for all its keys
                toks = {int(idx["entries"][rp[k]]) // (w.num_kv_heads * w.topk) for k in keys}
                assert len(toks) == 1 and tq[np.searchsorted(w.cu_seqlens_q, toks.pop(), side="right") - 1] == 1
            assert sorted(covered) == list(range(len(idx["entries"])))
            # the fewest items the size limits allow, split evenly: a normal
            # key of cnt entries gets ceil(cnt / E) items, a decode run of
            # len keys ceil(len / D), item sizes differing by at most one
            E = R * max(1, 128 // G)
            per_key = {}
            for key, _, n, _ in sch["items"]:
                per_key.setdefault(int(key), []).append(int(n))
            for key, sizes in per_key.items():
                cnt = int(rp[key + 1] - rp[key])
                assert sum(sizes) == cnt and len(sizes) == -(-cnt // E) and max(sizes) - min(sizes) <= 1
            per_run = {}
            for a0, e, _, nk in sch["items_dec"]:
                g = int(active[a0]) // idx["nb"]
                tok = int(idx["entries"][e]) // (w.num_kv_heads * w.topk)
                per_run.setdefault((tok, g), []).append(int(nk))
            for (tok, g), sizes in per_run.items():
                run = int(np.count_nonzero(idx["slot_entry"][(tok * w.num_kv_heads + g) * w.topk:
                                                             (tok * w.num_kv_heads + g + 1) * w.topk] >= 0))
                assert sum(sizes) == run and len(sizes) == -(-run // D) and max(sizes) - min(sizes) <= 1
            for it, cp, cost in (("items", "cta_ptr", "cost_prefix"), ("items_dec", "cta_ptr_dec", "cost_prefix_dec")):
                c = sch[cp]
                assert c[0] == 0 and c[-1] == len(sch[it]) and np.all(np.diff(c) >= 0)
                if len(sch[it]):
                    costs = np.diff(sch[cost])
                    C = sch[cost][-1]
                    for k in range(P):
                        assert costs[c[k]:c[k + 1]].sum() <= C / P + costs.max() + 1
            sch2 = oracle.schedule(prob, w.used_kv_lens, w.cu_seqlens_q, idx, R, D, P)
            assert all(np.array_equal(sch[k], sch2[k]) for k in sch)


# ----------------------------------------------------------- workload recipes
def test_workload_recipes():
    w = W.workload("gqa_decode")
    nblk = (w.used_kv_lens.astype(np.int64) + 127) // 128
    for t in range(w.total_q):
        for g in range(8):
            row = w.selected[t, g]
            assert row[0] == nblk[t] - 1 and len(set(row.tolist())) == 16 and row.min() >= 0
    w = W.workload("tiny_decode")
    assert w.used_kv_lens.tolist() == [256, 1024] and w.selected.shape == (2, 1, 2)
    assert sorted(np.unique(w.block_tables[w.block_tables >= 0]).tolist()) == list(range(w.num_pages))
