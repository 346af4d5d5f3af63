"""Pins of the oracle's physically keyed index (cross-sequence block dedup):
sequences that share a cached prefix point their block tables at the same
pages, and a block is then one key for every row of every sequence that
selected it.  Checked against a brute force written here over the
definition (block identity = logical block + physical pages, full blocks
only, owner = the smallest sequence), against the plain index when nothing
is shared, and by the property that makes dedup exact: every row of a key
reads the same pages at the same positions as its own block."""
import numpy as np
import pytest

import oracle
from block_sparse_attention_builder_gb300 import workloads as W

BLOCK = 128


def _shared(name, tq, lens, hq, hkv, ps, topk, causal, selection, seed):
    return W.custom(name, tq, lens, hq, hkv, ps, topk, causal, selection, seed,
                    extra={"shared_prefix_blocks": 64})


CASES = {
    # decode rows; hot sequences s and s + 16 of a group share their prefix
    "decode_ps64": _shared("dd64", [1] * 24, [9000, 3000, 700, 20000, 129, 8192] * 4, 16, 2, 64, 16, False,
                           "hot_groups", 140),
    # prefill rows, causal, page 128 (positions differ between the sharers)
    "prefill_ps128": _shared("dp128", [1, 3, 0, 5] * 6, [9000, 4000, 300, 12000] * 6, 8, 1, 128, 8, True,
                             "hot_groups", 141),
}


def _brute(w):
    """The definition, one slot at a time."""
    B, Hkv, K, ps = w.num_seqs, w.num_kv_heads, w.topk, w.page_size
    lens = [int(x) for x in w.used_kv_lens]
    nblk = [(L + BLOCK - 1) // BLOCK for L in lens]
    off = [0]
    for n in nblk:
        off.append(off[-1] + n)
    NB = off[-1]
    per = BLOCK // ps

    def pages(s, b):
        return tuple(int(w.block_tables[s, b * per + j]) for j in range(per))

    def shareable(s, b):
        return BLOCK * b + BLOCK <= lens[s] and all(0 <= pg < w.num_pages for pg in pages(s, b))

    def owner(s, b):
        if not shareable(s, b):
            return s
        for s2 in range(s):
            if b < nblk[s2] and shareable(s2, b) and pages(s2, b) == pages(s, b):
                return s2
        return s

    keys = []
    for t in range(w.total_q):
        s = int(np.searchsorted(w.cu_seqlens_q, t, side="right") - 1)
        Tq = int(w.cu_seqlens_q[s + 1] - w.cu_seqlens_q[s])
        pos = lens[s] - Tq + (t - int(w.cu_seqlens_q[s]))
        for g in range(Hkv):
            seen = set()
            for k in range(K):
                b = int(w.selected[t, g, k])
                slot = (t * Hkv + g) * K + k
                if b == -1 or b in seen or not (0 <= b < nblk[s]):
                    seen.add(b)
                    continue
                seen.add(b)
                if w.causal and BLOCK * b > pos:
                    continue
                keys.append((g * NB + off[owner(s, b)] + b, slot))
    keys.sort()
    row_ptr = np.zeros(Hkv * NB + 1, np.int64)
    for key, _ in keys:
        row_ptr[key + 1] += 1
    row_ptr = np.cumsum(row_ptr)
    entries = np.array([slot for _, slot in keys], np.int64)
    slot_entry = np.full(w.total_q * Hkv * K, -1, np.int64)
    slot_entry[entries] = np.arange(len(entries))
    return row_ptr, entries, slot_entry


@pytest.mark.parametrize("name", list(CASES))
def test_dedup_index_equals_brute_force(name):
    w = CASES[name]
    got = oracle.build_index_dedup(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens,
                                   w.block_tables)
    row_ptr, entries, slot_entry = _brute(w)
    assert got["flags"] == 0
    assert np.array_equal(got["row_ptr"], row_ptr)
    assert np.array_equal(got["entries"], entries)
    assert np.array_equal(got["slot_entry"], slot_entry)


@pytest.mark.parametrize("name", list(CASES))
def test_dedup_merges_rows_of_shared_blocks(name):
    """Sharing moves rows into fewer keys: the same slots are entries, and
    keys gain rows from more than one sequence."""
    w = CASES[name]
    prob = oracle.problem_for(w)
    plain = oracle.build_index(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens)
    dedup = oracle.build_index_dedup(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens, w.block_tables)
    assert np.array_equal(np.sort(plain["entries"]), np.sort(dedup["entries"]))
    assert np.count_nonzero(np.diff(dedup["row_ptr"])) < np.count_nonzero(np.diff(plain["row_ptr"]))
    Hkv, K = w.num_kv_heads, w.topk
    seq_of = lambda slot: int(np.searchsorted(w.cu_seqlens_q, slot // (Hkv * K), side="right") - 1)
    counts = np.diff(dedup["row_ptr"])
    multi = [k for k in np.nonzero(counts)[0]
             if len({seq_of(e) for e in dedup["entries"][dedup["row_ptr"][k]:dedup["row_ptr"][k + 1]]}) > 1]
    assert multi


@pytest.mark.parametrize("name", list(CASES))
def test_every_row_of_a_key_reads_its_own_pages(name):
    """What makes dedup exact: for every entry, the key's block (owner
    sequence, logical block) has the same pages and the same 128 valid
    tokens as the block the row selected in its own sequence."""
    w = CASES[name]
    Hkv, K, ps = w.num_kv_heads, w.topk, w.page_size
    per = BLOCK // ps
    idx = oracle.build_index_dedup(oracle.problem_for(w), w.selected, w.cu_seqlens_q, w.used_kv_lens,
                                   w.block_tables)
    lens = w.used_kv_lens.astype(np.int64)
    nblk = (lens + BLOCK - 1) // BLOCK
    off = np.concatenate([[0], np.cumsum(nblk)])
    NB = int(off[-1])
    for key in np.nonzero(np.diff(idx["row_ptr"]))[0]:
        r = int(key % NB)
        ks = int(np.searchsorted(off, r, side="right") - 1)
        kb = r - int(off[ks])
        for e in idx["entries"][idx["row_ptr"][key]:idx["row_ptr"][key + 1]]:
            t, g, k = e // (Hkv * K), (e // K) % Hkv, e % K
            s = int(np.searchsorted(w.cu_seqlens_q, t, side="right") - 1)
            b = int(w.selected[t, g, k])
            assert b == kb and g == key // NB
            if s != ks:
                assert ks < s
                assert BLOCK * (b + 1) <= min(lens[s], lens[ks])
                assert np.array_equal(w.block_tables[s, b * per:(b + 1) * per],
                                      w.block_tables[ks, b * per:(b + 1) * per])


def test_without_shared_pages_dedup_is_the_plain_index():
    for w in (W.custom("np1", [1] * 20, [5000, 300, 129] * 6 + [64, 9000], 16, 2, 64, 8, False, "hot_groups", 142),
              W.custom("np2", [2, 0, 7, 1], [700, 128, 2000, 5000], 8, 1, 128, 6, True, "uniform", 143),
              W.workload("tiny_decode")):
        prob = oracle.problem_for(w)
        a = oracle.build_index(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens)
        b = oracle.build_index_dedup(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens, w.block_tables)
        for k in a:
            assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k


def test_partial_and_invalid_blocks_are_never_shared():
    """Two sequences whose tables name the same pages for a partial last
    block, or for a block with an out-of-range page, keep separate keys."""
    w = W.custom("pp", [1, 1], [200, 200], 8, 1, 64, 2, False, "all", 144)
    w.block_tables[1, :] = w.block_tables[0, :]  # block 0 full and shared, block 1 partial (72 tokens)
    prob = oracle.problem_for(w)
    idx = oracle.build_index_dedup(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens, w.block_tables)
    counts = np.diff(idx["row_ptr"])
    # keys: (s0,b0) (s0,b1) (s1,b0) (s1,b1): block 0 merged, block 1 not
    assert counts.tolist() == [2, 1, 0, 1]
    w.block_tables[:, 1] = w.num_pages + 5    # block 0's second page out of range: not shareable
    idx = oracle.build_index_dedup(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens, w.block_tables)
    assert np.diff(idx["row_ptr"]).tolist() == [1, 1, 1, 1]


def test_shared_prefix_page_tables_recipe():
    """The generator's shared-prefix tables: hot sequence s + 16 points the
    pages of each block that is full in both at sequence s's pages (the
    group's first hot sequence), for the first 64 blocks, and nothing else
    changes (the selections and the other rows are those of the plain
    recipe)."""
    lens = [9000, 3000, 700, 20000, 129, 8192] * 4
    plain = W.custom("r0", [1] * 24, lens, 16, 2, 64, 16, False, "hot_groups", 150)
    shared = W.custom("r0", [1] * 24, lens, 16, 2, 64, 16, False, "hot_groups", 150,
                      extra={"shared_prefix_blocks": 64})
    assert np.array_equal(plain.selected, shared.selected)
    per = BLOCK // 64
    for s in range(24):
        hot = (s // 8) % 2 == 0
        if not hot or s < 8:  # cold sequences and each group's first hot sequence keep their pages
            assert np.array_equal(plain.block_tables[s], shared.block_tables[s]), s
            continue
        o = s - 16
        full = min(lens[s], lens[o]) // BLOCK
        n = min(64, full) * per
        assert np.array_equal(shared.block_tables[s, :n], shared.block_tables[o, :n])
        assert np.array_equal(shared.block_tables[s, n:], plain.block_tables[s, n:])


@pytest.mark.parametrize("name", list(CASES))
def test_block_owners_equal_brute_force(name):
    """The owner map on its own (the table the dedup index is keyed by)."""
    w = CASES[name]
    ps, per = w.page_size, BLOCK // w.page_size
    lens = [int(x) for x in w.used_kv_lens]
    nblk = [(L + BLOCK - 1) // BLOCK for L in lens]

    def pages(s, b):
        return tuple(int(w.block_tables[s, b * per + j]) for j in range(per))

    def shareable(s, b):
        return BLOCK * b + BLOCK <= lens[s] and all(0 <= pg < w.num_pages for pg in pages(s, b))

    want = []
    for s in range(w.num_seqs):
        for b in range(nblk[s]):
            o = s
            if shareable(s, b):
                o = next(s2 for s2 in range(s + 1) if b < nblk[s2] and shareable(s2, b) and pages(s2, b) == pages(s, b))
            want.append(o)
    got = oracle.block_owners(oracle.problem_for(w), w.used_kv_lens, w.block_tables)
    assert got.tolist() == want
    assert any(o != s for o, s in zip(got, np.repeat(np.arange(w.num_seqs), nblk)))  # something is shared


def test_schedule_of_a_dedup_index_worked_example():
    """Hand-worked schedule of a deduplicated decode batch.  Two sequences of
    one new token each, L = 512 (4 blocks), Hkv 1, G 16, page 128; sequence
    1's blocks 0 and 1 sit on sequence 0's pages; both select blocks 0..3.
    Dedup index (key = g*NB + blk_off[owner] + b, NB = 8):
      key 0 (s0 b0): 2 entries (both tokens), key 1 (s0 b1): 2 entries,
      key 2 (s0 b2): token 0, key 3 (s0 b3): token 0,
      keys 4, 5 (s1 b0, b1): none, key 6 (s1 b2): token 1, key 7 (s1 b3): token 1.
    Keys 0 and 1 hold two entries, so they are NORMAL (one item each);
    keys 2, 3 and 6, 7 are decode keys forming two runs of two."""
    prob = oracle.problem(2, 2, 16, 1, 4, 128, 8, 4, False)
    bt = np.array([[0, 1, 2, 3], [0, 1, 6, 7]], dtype=np.int32)
    lens = np.array([512, 512], dtype=np.int32)
    cu = np.array([0, 1, 2], dtype=np.int64)
    sel = np.array([[[0, 1, 2, 3]], [[3, 2, 1, 0]]], dtype=np.int32)
    idx = oracle.build_index_dedup(prob, sel, cu, lens, bt)
    # slots: token t, slot k -> t * 4 + k
    assert list(idx["row_ptr"]) == [0, 2, 4, 5, 6, 6, 6, 7, 8]
    assert list(idx["entries"]) == [0, 7, 1, 6, 2, 3, 5, 4]
    sch = oracle.schedule(prob, lens, cu, idx, 4, 8, 2)
    # normal: cost 384 + 128 * 2 (bf16) + 1 tile * 256 + 2 rows-of-16 * 3 = 992
    assert sch["items"].tolist() == [[0, 0, 2, 0], [1, 2, 2, 0]]
    assert sch["cost_prefix"].tolist() == [0, 992, 1984]
    # decode: {active position, entry, 1, keys}; cost 2 * 64 + 256 + 2 * 128 * 2 = 896
    assert sch["items_dec"].tolist() == [[2, 4, 1, 2], [4, 6, 1, 2]]
    assert sch["cost_prefix_dec"].tolist() == [0, 896, 1792]
