"""CPU-side checks of the C ABI: the library builds, loads without a GPU and
exports every symbol include/mxsa.h declares; host-side validation and
workspace sizing behave as documented (no compute calls here)."""
import ctypes
import os
import re

import pytest
import torch

import block_sparse_attention_builder_gb300 as mx
from block_sparse_attention_builder_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return mx.library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "mxsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mxsa_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert "mxsa_kvouter_fwd" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(mx.EXPORTED) | set(names)


def test_test_switch_only_in_the_test_library(lib):
    """The barrier switch of the wait-limit test exists only in the
    separate test library, never in libmxsa.so."""
    assert not hasattr(lib, "mxsa_test_skip_barrier_arrival")
    test_lib = mx._load_library(B.TEST_LIB)
    assert hasattr(test_lib, "mxsa_test_skip_barrier_arrival")


def test_version_and_status_strings(lib):
    assert lib.mxsa_version() >> 16 == 1
    for code, name in mx.STATUS_NAMES.items():
        assert lib.mxsa_status_string(code).decode() == name


def _prob(**kw):
    base = dict(num_seqs=2, total_q=4, num_q_heads=16, num_kv_heads=2, topk=8, page_size=64, num_pages=100,
                max_pages_per_seq=40, causal=False)
    base.update(kw)
    return mx.make_problem(**base)


def test_workspace_sizes_are_shape_upper_bounds(lib):
    p = _prob()
    ib, sb, pb = mx.workspace_size(p)
    L = mx.index_layout(p)
    assert ib == L.total and L.nslots == 4 * 2 * 8
    assert L.keys_cap == 2 * 2 * 20  # Hkv * B * ceil(40 * 64 / 128)
    assert pb >= L.nslots * 8 * (128 * 2 + 4)  # one 16-bit row + an FP32 lse per (slot, head)
    pf = mx.workspace_size(_prob(kv_dtype=torch.float8_e4m3fn))[2]
    assert pf >= L.nslots * 8 * (128 * 4 + 4)  # FP8 caches: FP32 rows
    S = mx.sched_layout(p)
    assert sb == S.total and S.items_cap == L.nslots
    offs = [L.header, L.seq_info, L.token_seq, L.slot_entry, L.bitmap, L.kmap, L.counts, L.row_ptr, L.entries,
            L.active_keys, L.active_valid, L.row_nnz, L.row_minb, L.row_maxb, L.cta_sums, L.total]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(page_size=32), 2), (dict(num_q_heads=12, num_kv_heads=5), 1),
    (dict(num_q_heads=256, num_kv_heads=1), 2), (dict(topk=300), 2), (dict(topk=0), 1), (dict(num_seqs=0), 1),
    (dict(num_pages=0), 1), (dict(causal=2), 1), (dict(softmax_scale=-1.0), 1),
])
def test_invalid_problems_are_rejected(lib, kw, status):
    p = _prob()
    for k, v in kw.items():
        setattr(p, k, v)
    with pytest.raises(mx.MxsaError) as ei:
        mx.workspace_size(p)
    assert ei.value.status == status


def test_unsupported_dtype_pairs(lib):
    p = _prob(q_dtype=torch.bfloat16, kv_dtype=torch.float16)
    with pytest.raises(mx.MxsaError) as ei:
        mx.workspace_size(p)
    assert ei.value.status == 2
    p = _prob(q_dtype=torch.float16, kv_dtype=torch.float8_e4m3fn)
    assert mx.workspace_size(p)[0] > 0


def test_null_and_small_workspace_rejected_before_any_launch(lib):
    p = _prob()
    ib, sb, pb = mx.workspace_size(p)
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    assert lib.mxsa_build_index(ctypes.byref(p), fake, None, fake, fake, ib, None) == 1
    assert lib.mxsa_build_index(ctypes.byref(p), fake, fake, fake, fake, ib - 1, None) == 3
    assert lib.mxsa_build_index(ctypes.byref(p), P((1 << 20) + 2), fake, fake, fake, ib, None) == 1
    assert lib.mxsa_schedule(ctypes.byref(p), fake, ib, 0, fake, sb - 256, None) == 3
    assert lib.mxsa_schedule(ctypes.byref(p), fake, ib, 5000, fake, sb, None) == 1
    assert lib.mxsa_kvouter_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, ib, fake, sb, 1, fake, pb - 1,
                                None) == 3
    assert lib.mxsa_combine(ctypes.byref(p), fake, ib, fake, pb, P((1 << 20) + 8), None, None) == 1
    assert lib.mxsa_read_status(None, None, None) == 1
    assert lib.mxsa_workspace_size(None, None, None, None) == 1


def test_package_has_no_cpu_fallback():
    import block_sparse_attention_builder_gb300 as pkg
    src = open(pkg.__file__).read()
    assert "import oracle" not in src and "from oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "block_sparse_attention_builder_gb300", "csrc")):
        text = open(os.path.join(ROOT, "block_sparse_attention_builder_gb300", "csrc", f)).read()
        assert "oracle" not in text.lower() or f.endswith(".md")


def test_store_kv_arguments_rejected_before_any_launch(lib):
    P = ctypes.c_void_p
    fake, fake8 = P(1 << 20), P((1 << 20) + 8)  # never dereferenced: validation fails first
    p = _prob(kv_dtype=torch.float8_e4m3fn)
    ok_args = [fake, fake, fake, fake, fake]
    # a cache dtype that is neither the source's nor e4m3
    bad = _prob(q_dtype=torch.float16, kv_dtype=torch.bfloat16)
    assert lib.mxsa_store_kv(ctypes.byref(bad), 4, *ok_args, None, None, 0, 0, None, None) in (1, 2)
    assert lib.mxsa_store_kv(ctypes.byref(p), -1, *ok_args, None, None, 0, 0, None, None) == 1
    # index keys: both pointers or neither; dim a multiple of 8
    assert lib.mxsa_store_kv(ctypes.byref(p), 4, *ok_args, fake, None, 1, 64, None, None) == 1
    assert lib.mxsa_store_kv(ctypes.byref(p), 4, *ok_args, fake, fake, 1, 60, None, None) == 1
    assert lib.mxsa_store_kv(ctypes.byref(p), 4, *ok_args, fake, fake, 0, 64, None, None) == 1
    # null or misaligned tensors
    assert lib.mxsa_store_kv(ctypes.byref(p), 4, None, fake, fake, fake, fake, None, None, 0, 0, None, None) == 1
    assert lib.mxsa_store_kv(ctypes.byref(p), 4, fake, fake8, fake, fake, fake, None, None, 0, 0, None, None) == 1
    assert lib.mxsa_store_kv(None, 4, *ok_args, None, None, 0, 0, None, None) == 1


def test_dense_fwd_arguments_rejected_before_any_launch(lib):
    P = ctypes.c_void_p
    fake, fake8 = P(1 << 20), P((1 << 20) + 8)  # never dereferenced: validation fails first
    tabs = [fake, fake, fake]                      # block_tables, cu_seqlens_q, used_kv_lens
    p = _prob()

    def call(prob, q=fake, k=fake, v=fake, t=tabs, out=fake, lse=None, flags=None):
        pr = ctypes.byref(prob) if prob is not None else None
        return lib.mxsa_dense_fwd(pr, q, k, v, *t, out, lse, flags, None)

    assert call(None) == 1
    # the caches must hold the query's type (no FP8 widening on this path)
    assert call(_prob(kv_dtype=torch.float8_e4m3fn)) == 2
    assert call(_prob(num_seqs=1025)) == 2  # the sequence table lives in shared memory
    assert call(_prob(num_q_heads=12, num_kv_heads=5)) == 1  # an invalid shape stays invalid here
    # topk is not the dense path's: a problem whose slot count the sparse
    # index could not hold still passes validation (a null q is the error)
    big = _prob(total_q=1 << 24, num_kv_heads=2, num_q_heads=16, topk=256)
    assert lib.mxsa_workspace_size(ctypes.byref(big), None, None, None) in (1, 2)
    assert call(big, q=None) == 1 and call(_prob(topk=0), q=None) == 1
    # null tables; null tensors while there are tokens
    assert call(p, t=[None, fake, fake]) == 1
    assert call(p, t=[fake, fake, None]) == 1
    assert call(p, q=None) == 1
    assert call(p, out=None) == 1
    # misaligned tensors and tables
    assert call(p, q=fake8) == 1
    assert call(p, t=[P((1 << 20) + 2), fake, fake]) == 1
    assert call(p, t=[fake, P((1 << 20) + 4), fake]) == 1
    assert call(p, lse=P((1 << 20) + 2)) == 1


def test_binding_refuses_buffers_smaller_than_the_problem(lib):
    """A pointer carries no size, so the binding compares every tensor's
    bytes with what the problem's shape makes the kernels touch, and refuses
    short or non-contiguous tensors before the C call (no GPU needed: the
    refusal comes first)."""
    p = _prob(num_seqs=2, total_q=4, num_q_heads=16, num_kv_heads=2, topk=8, page_size=64, num_pages=100,
              max_pages_per_seq=40)
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    q, out = bf(4, 16, 128), bf(4, 16, 128)
    kc = torch.zeros(100 * 2 * 64 * 128 * 2, dtype=torch.uint8)  # raw bytes are accepted
    bt = torch.zeros(2, 40, dtype=torch.int32)
    cu, lens = torch.zeros(3, dtype=torch.int64), torch.zeros(2, dtype=torch.int32)
    lse = torch.zeros(16, 4, dtype=torch.float32)
    sel = torch.zeros(4, 2, 8, dtype=torch.int32)
    ws = torch.zeros(16, dtype=torch.uint8)

    def refused(fn, *a, **k):
        with pytest.raises(mx.MxsaError) as ei:
            fn(*a, **k)
        assert ei.value.status == 1

    refused(mx.dense_fwd, p, q[:3], kc, kc, bt, cu, lens, out, lse)          # q short by one token
    refused(mx.dense_fwd, p, q, kc[:-1], kc, bt, cu, lens, out, lse)         # cache short by one byte
    refused(mx.dense_fwd, p, q, kc, kc, bt[:, :39], cu, lens, out, lse)      # table narrower than max_pages
    refused(mx.dense_fwd, p, q, kc, kc, bt, cu[:2], lens, out, lse)          # cu_seqlens_q needs B + 1
    refused(mx.dense_fwd, p, q, kc, kc, bt, cu, lens, out, lse[:, :3])       # lse short
    refused(mx.dense_fwd, p, q, kc, kc, bt, cu, lens, out.transpose(0, 1), lse)  # not contiguous
    refused(mx.plan, p, sel[:, :, :7].contiguous(), cu, lens, ws, ws)        # topk slots short
    refused(mx.build_index, p, sel, cu, lens[:1], ws)
    refused(mx.kvouter_fwd, p, q, kc, kc[:10], bt, ws, ws, ws)
    refused(mx.combine, p, ws, ws, out[:2])
    ps = _prob(num_q_heads=2, num_kv_heads=2, page_size=64, num_pages=3, kv_dtype=torch.float8_e4m3fn)
    loc = torch.zeros(5, dtype=torch.int64)
    k5 = bf(5, 2, 128)
    c8 = torch.zeros(3, 2, 64, 128, dtype=torch.uint8)
    refused(mx.store_kv, ps, loc, k5[:4], k5, c8, c8)                        # k short
    refused(mx.store_kv, ps, loc, k5, k5, c8[:2], c8)                        # cache short
    refused(mx.store_kv, ps, loc, k5, k5, c8, c8, idx_k=bf(5, 1, 64),
            idx_cache=torch.zeros(3, 1, 64, 63, dtype=torch.uint8))          # index cache short
