"""Pins of the oracle's top-k block selection (oracle.select_blocks).

The pages name the step ("sparse top-k selection" over an index K cache)
but not its scoring rule; the reading the oracle states is: a block's score
is the largest FP32 dot product (fused multiply-adds in dimension order)
of the token's index query with the index keys of its visible positions,
and the top-k blocks by (score descending, block ascending) are selected,
-1 filling the rest.  Each part is pinned here by something other than the
oracle itself:
  - the scores against float64 dot products computed by numpy from torch's
    own decoding, within the FP32 summation bound, with NaN exactly where a
    block has no visible position;
  - the ranking against Python's sort of the oracle's own scores, and the
    selected set against the exact float64 scores;
  - closed cases: equal blocks (ties), a huge key at the row's own causal
    position and one just past it, keys past the sequence's length, invalid
    pages, NaN keys, fewer valid blocks than top-k, and a shuffled page
    table (the same result).
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_builder_gb300 import workloads as W

U32 = 2.0 ** -24


def _case(name, tq, lens, hkv, ps, topk, causal, dtype, seed, dim=64):
    w = W.custom(name, tq, lens, hkv * 2, hkv, ps, topk, causal, "uniform", seed, q_dtype="bf16" if dtype == "fp8" else dtype,
                 kv_dtype=dtype)
    return w, w.idx_q(dim), w.idx_cache(dim)


def _prob(w):
    return oracle.problem_for(w)


def _select(w, dim, iq, ik, bt=None, with_scores=True):
    return oracle.select_blocks(_prob(w), dim, iq, ik, w.block_tables if bt is None else bt, w.cu_seqlens_q,
                                w.used_kv_lens, with_scores=with_scores, nthreads=4)


def exact_scores(w, iq, ik, bt=None):
    """float64 block maxima and their FP32 summation bounds, from the
    definition, one position at a time."""
    bt = w.block_tables if bt is None else bt
    q = iq.float().double().numpy()
    k = ik.float().double().numpy()
    T, H, D = q.shape
    ps = w.page_size
    nbm = (w.max_pages_per_seq * ps + 127) // 128
    best = np.full((T, H, nbm), np.nan)
    bound = np.zeros((T, H, nbm))
    cap = w.max_pages_per_seq * ps
    for s in range(w.num_seqs):
        L = min(max(int(w.used_kv_lens[s]), 0), cap)
        t0, t1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
        for t in range(t0, t1):
            pos = L - (t1 - t0) + (t - t0)
            for g in range(H):
                for b in range((L + 127) // 128):
                    for p in range(128 * b, min(128 * b + 128, L)):
                        if w.causal and p > pos:
                            break
                        page = int(bt[s, p // ps])
                        if page < 0 or page >= w.num_pages:
                            continue
                        prod = q[t, g] * k[page, g, p % ps]
                        d = float(prod.sum())
                        if np.isnan(d):
                            continue
                        if np.isnan(best[t, g, b]) or d > best[t, g, b]:
                            best[t, g, b] = d
                        bound[t, g, b] = max(bound[t, g, b], D * U32 * float(np.abs(prod).sum()) * 1.01)
    return best, bound


def ranking_from_scores(scores, topk):
    """Python's sort of a row's block scores: (score descending, block
    ascending), NaN = no score, -1 fill."""
    T, H, nb = scores.shape
    sel = np.full((T, H, topk), -1, np.int32)
    for t in range(T):
        for g in range(H):
            ok = [(0.0 if v == 0 else float(v), b) for b, v in enumerate(scores[t, g]) if not np.isnan(v)]
            ok.sort(key=lambda x: (-x[0], x[1]))
            for i, (_, b) in enumerate(ok[:topk]):
                sel[t, g, i] = b
    return sel


CASES = [
    ("dec_fp8", [1, 1, 1], [300, 1000, 129], 2, 64, 4, False, "fp8", 11),
    ("pre_fp8", [5, 9], [700, 1300], 1, 128, 6, True, "fp8", 12),
    ("pre_bf16", [3, 17], [500, 2100], 2, 64, 5, True, "bf16", 13),
    ("mixed_fp16", [1, 6, 2], [1200, 900, 260], 2, 128, 3, True, "fp16", 14),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_scores_match_float64_definition(case):
    w, iq, ik = _case(*case)
    _, got = _select(w, 64, iq, ik)
    ref, bound = exact_scores(w, iq, ik)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "blocks with a score differ"
    fin = ~np.isnan(ref)
    err = np.abs(got[fin].astype(np.float64) - ref[fin])
    assert np.all(err <= bound[fin] + 1e-30), f"max excess {np.max(err - bound[fin]):.3g}"


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ranking_and_selected_set(case):
    w, iq, ik = _case(*case)
    sel, scores = _select(w, 64, iq, ik)
    assert np.array_equal(sel, ranking_from_scores(scores, w.topk))
    # the selected blocks are the best by the exact scores (up to the bound)
    ref, bound = exact_scores(w, iq, ik)
    T, H, K = sel.shape
    for t in range(T):
        for g in range(H):
            chosen = [b for b in sel[t, g] if b >= 0]
            rest = [b for b in range(ref.shape[2]) if not np.isnan(ref[t, g, b]) and b not in chosen]
            if chosen and rest:
                lo = min(ref[t, g, b] - bound[t, g, b] for b in chosen)
                hi = max(ref[t, g, b] + bound[t, g, b] for b in rest)
                assert lo <= hi or lo >= max(ref[t, g, b] for b in rest) - 1e-30
                assert min(ref[t, g, b] for b in chosen) >= max(ref[t, g, b] for b in rest) - 2 * max(
                    bound[t, g].max(), 1e-30)


def _bits8(x):
    return x.view(torch.uint8) if x.element_size() == 1 else x.view(torch.int16)


def test_equal_blocks_rank_the_smaller_first():
    w, iq, ik = _case("ties", [1], [1024], 1, 128, 8, False, "fp8", 21)
    ik = ik.clone()
    bt = w.block_tables
    # blocks 5 and 2 get block 6's keys: three equal scores
    for dst in (5, 2):
        ik[int(bt[0, dst])] = ik[int(bt[0, 6])]
    sel, scores = _select(w, 64, iq, ik)
    assert scores[0, 0, 2] == scores[0, 0, 5] == scores[0, 0, 6]
    order = [b for b in sel[0, 0] if b in (2, 5, 6)]
    assert order == [2, 5, 6]


def test_causal_position_is_visible_and_the_next_is_not():
    # one sequence of 4 new tokens on L = 300: token i sits at position 296 + i
    w, iq, ik = _case("causal", [4], [300], 1, 128, 3, True, "fp8", 22)
    ik = ik.clone()
    iq = iq.clone()
    one = torch.tensor(1.0).to(iq.dtype)
    iq[:] = torch.zeros((), dtype=iq.dtype)
    iq[:, :, 0] = one
    ik[:] = torch.zeros((), dtype=ik.dtype)
    big = torch.tensor(448.0).to(ik.dtype)
    p = 297  # token 1's own position; token 0 must not see it
    ik[int(w.block_tables[0, p // 128]), 0, p % 128, 0] = big
    sel, scores = _select(w, 64, iq, ik)
    assert scores[1, 0, 2] == 448.0 and sel[1, 0, 0] == 2
    assert scores[0, 0, 2] == 0.0  # positions 256..296 only


def test_positions_past_the_length_and_on_bad_pages_are_skipped():
    w, iq, ik = _case("len", [1, 1], [200, 384], 1, 64, 4, False, "fp8", 23)
    ik = ik.clone()
    iq = iq.clone()
    iq[:] = torch.zeros((), dtype=iq.dtype)
    iq[:, :, 0] = torch.tensor(1.0).to(iq.dtype)
    ik[:] = torch.zeros((), dtype=ik.dtype)
    big = torch.tensor(448.0).to(ik.dtype)
    # sequence 0 (L = 200): position 230 lies in the page of 192..255 but past L
    ik[int(w.block_tables[0, 230 // 64]), 0, 230 % 64, 0] = big
    sel, scores = _select(w, 64, iq, ik)
    assert scores[0, 0, 1] == 0.0 and (np.isnan(scores[0, 0, 2:])).all()
    # sequence 1: a bad page makes its positions invisible; a block whose
    # pages are all bad has no score and is never selected
    bt = w.block_tables.copy()
    bt[1, 2] = -1
    bt[1, 3] = w.num_pages + 5
    sel, scores = _select(w, 64, iq, ik, bt=bt)
    assert np.isnan(scores[1, 0, 1]) and 1 not in sel[1, 0]
    assert list(sel[1, 0]) == [0, 2, -1, -1]


def test_nan_keys_are_skipped_and_topk_beyond_the_blocks_is_padded():
    w, iq, ik = _case("nan", [1], [256], 1, 128, 5, False, "fp8", 24)
    ik = ik.clone()
    raw = ik.view(torch.uint8)
    page0 = int(w.block_tables[0, 0])
    raw[page0] = 0x7F  # every key of block 0 is NaN in every dimension
    sel, scores = _select(w, 64, iq, ik)
    assert np.isnan(scores[0, 0, 0]) and not np.isnan(scores[0, 0, 1])
    assert list(sel[0, 0]) == [1, -1, -1, -1, -1]


def test_shuffled_pages_give_the_same_selection():
    w, iq, ik = _case("perm", [1, 3], [900, 700], 2, 64, 4, True, "bf16", 25)
    sel, _ = _select(w, 64, iq, ik, with_scores=True)
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.num_pages)  # physical page p moves to perm[p]
    ik2 = torch.empty_like(ik)
    ik2[torch.from_numpy(perm)] = ik
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    sel2, _ = _select(w, 64, iq, ik2, bt=bt2)
    assert np.array_equal(sel, sel2)
