"""Helpers for the GPU tests: run the library's four steps through the C ABI
on a generated workload, read its workspaces back, and build the oracle's
expected values (oracle calls only -- nothing here comes from the GPU path).
"""
import numpy as np
import torch

import block_sparse_attention_builder_gb300 as mx
import oracle

TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.float8_e4m3fn}
ITEM_TILES = 4
DECODE_BLOCKS = 8


def device_inputs(w, device="cuda"):
    return dict(
        q=w.q(device), k=w.k_cache(device), v=w.v_cache(device),
        sel=torch.from_numpy(w.selected).to(device), bt=torch.from_numpy(w.block_tables).to(device),
        cu=torch.from_numpy(w.cu_seqlens_q).to(device), lens=torch.from_numpy(w.used_kv_lens).to(device))


def problem(w, scale=0.0):
    kv = "nvfp4" if w.spec.kv_dtype == "nvfp4" else TORCH[w.spec.kv_dtype]
    return mx.make_problem(w.num_seqs, w.total_q, w.num_q_heads, w.num_kv_heads, w.topk, w.page_size, w.num_pages,
                           w.max_pages_per_seq, w.causal, scale, TORCH[w.spec.q_dtype], kv)


def run(w, inp=None, num_ctas=0, scale=0.0):
    inp = inp or device_inputs(w)
    prob = problem(w, scale)
    attn = mx.SparseAttention(prob, "cuda", num_ctas)
    out, lse = attn(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"])
    torch.cuda.synchronize()
    return attn, out, lse, inp


def read_index(attn):
    L = mx.index_layout(attn.prob)
    ws = attn.ws.index.cpu().numpy()
    i32 = lambda off, n: ws[off:off + 4 * n].view(np.int32).copy()
    hdr = i32(L.header, 16)
    flags, nb, nnz, n_active, n_keys = (int(x) for x in hdr[:5])
    return dict(flags=flags, nb=nb, nnz=nnz, n_active=n_active, n_keys=n_keys,
                row_ptr=i32(L.row_ptr, n_keys + 1), entries=i32(L.entries, nnz),
                slot_entry=i32(L.slot_entry, int(L.nslots)), active=i32(L.active_keys, n_active))


def read_sched(attn, num_ctas):
    L = mx.sched_layout(attn.prob)
    ws = attn.ws.sched.cpu().numpy()
    hdr = ws[L.header:L.header + 64].view(np.int32)
    n, nd = int(hdr[0]), int(hdr[5])
    items = ws[L.items:L.items + 16 * n].view(np.int32).reshape(n, 4).copy()
    cost = ws[L.cost_prefix:L.cost_prefix + 8 * (n + 1)].view(np.int64).copy()
    cta = ws[L.cta_ptr:L.cta_ptr + 4 * (num_ctas + 1)].view(np.int32).copy()
    items_d = ws[L.items_dec:L.items_dec + 16 * nd].view(np.int32).reshape(nd, 4).copy()
    cost_d = ws[L.cost_prefix_dec:L.cost_prefix_dec + 8 * (nd + 1)].view(np.int64).copy()
    cta_d = ws[L.cta_ptr_dec:L.cta_ptr_dec + 4 * (num_ctas + 1)].view(np.int32).copy()
    return dict(items=items, cost_prefix=cost, cta_ptr=cta, items_dec=items_d, cost_prefix_dec=cost_d,
                cta_ptr_dec=cta_d, num_ctas=int(hdr[1]))


def oracle_schedule(w, num_ctas):
    prob = oracle.problem_for(w)
    idx = oracle.build_index(prob, w.selected, w.cu_seqlens_q, w.used_kv_lens)
    return oracle.schedule(prob, w.used_kv_lens, w.cu_seqlens_q, idx, ITEM_TILES, DECODE_BLOCKS, num_ctas)


def partial_elem(prob):
    """Partial rows are FP32 with FP8 and NVFP4 caches, else the 16-bit q dtype."""
    return (torch.float32, 4) if prob.kv_dtype in (mx.FP8_E4M3, mx.NVFP4) else (mx._CODE_DTYPE[prob.q_dtype], 2)


def read_partials(attn):
    """Partial rows (o [nslots * G, 128] as float, lse [nslots * G]) of the
    partial workspace: the o rows, then the lses at a 256-byte boundary."""
    p = attn.prob
    G = p.num_q_heads // p.num_kv_heads
    nslots = p.total_q * p.num_kv_heads * p.topk
    n_o = nslots * G * 128
    dt, es = partial_elem(p)
    lse_off = ((n_o * es + 255) // 256) * 256
    ws = attn.ws.partial
    o = ws[:n_o * es].view(dt).float().view(nslots * G, 128).cpu().numpy()
    lse = ws[lse_off:lse_off + nslots * G * 4].view(torch.float32).cpu().numpy()
    return o, lse


def write_partials(attn, o, lse):
    """Writes partial rows o [nslots * G, 128] (rounded to the partial type)
    and lse [nslots * G] into the partial workspace, in read_partials' layout."""
    p = attn.prob
    G = p.num_q_heads // p.num_kv_heads
    nslots = p.total_q * p.num_kv_heads * p.topk
    n_o = nslots * G * 128
    dt, es = partial_elem(p)
    lse_off = ((n_o * es + 255) // 256) * 256
    part = attn.ws.partial
    ot = torch.from_numpy(np.asarray(o, np.float32).reshape(-1)).to(dt)
    part[:n_o * es].view(dt).copy_(ot)
    part[lse_off:lse_off + nslots * G * 4].view(torch.float32).copy_(torch.from_numpy(np.asarray(lse, np.float32)))


def oracle_full(w, rows=None):
    """Oracle (out [n,128], lse [n]) for rows t*Hq+h (all rows when None)."""
    prob = oracle.problem_for(w)
    if rows is None:
        return oracle.attention_rows(prob, w.q(), w.k_cache(), w.v_cache(), w.selected, w.block_tables,
                                     w.cu_seqlens_q, w.used_kv_lens)
    kc, vc, bt = w.compact_cache_for_rows(rows)
    prob.num_pages = max(1, kc.shape[0])
    q = w.q()
    return oracle.attention_rows(prob, q, kc, vc, w.selected, bt, w.cu_seqlens_q, w.used_kv_lens, rows=rows)


def oracle_slot_partials(w):
    """Per selection slot (t, g, k): the oracle's attention over that slot's
    block alone, for each of the G heads -> (o [nslots*G,128], lse [nslots*G])."""
    prob = oracle.problem_for(w)
    G = w.num_q_heads // w.num_kv_heads
    T, Hkv, K = w.selected.shape
    o = np.zeros((T, Hkv, K, G, 128))
    l = np.full((T, Hkv, K, G), -np.inf)
    q, kc, vc = w.q(), w.k_cache(), w.v_cache()
    for k in range(K):
        sel = np.full_like(w.selected, -1)
        sel[:, :, 0] = w.selected[:, :, k]
        ok, lk = oracle.attention_rows(prob, q, kc, vc, sel, w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
        o[:, :, k] = ok.reshape(T, Hkv, G, 128)
        l[:, :, k] = lk.reshape(T, Hkv, G)
    return o.reshape(-1, 128), l.reshape(-1)


def assert_close_out(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref) - (tol + tol * np.abs(ref))
    bad = err > 0
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance {tol}; first at {tuple(i)}: "
                             f"got {got[tuple(i)]} ref {ref[tuple(i)]}; max|d| {np.abs(got - ref).max():.3g}")


def assert_close_lse(got, ref, atol=2e-3, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)), f"{what}: lse finiteness differs"
    assert np.all(got[~fin] == ref[~fin]), f"{what}: infinite lse differs"
    if fin.any():
        d = np.abs(got[fin] - ref[fin]).max()
        assert d <= atol, f"{what}: lse max |d| {d:.3g} > {atol}"


def out_tol(w):
    return 4e-2 if w.spec.kv_dtype == "fp8" else 1e-2
