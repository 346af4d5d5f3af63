"""The allocation-free entry point, mxsa_attention_noalloc.

Some callers may not allocate device memory themselves: plug-ins inside a
host runtime that plans every buffer up front, or hot loops that must not
risk the device-wide synchronisation of a cudaMalloc/cudaFree.  For them the
library keeps its scratch in one fixed device array.  This test calls that
entry point through the C ABI twice in a row (two different problems, so the
second call runs on scratch the first one left behind) and compares each
result with the regular four-step entry points.  The file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_attention_builder_gb300 as mx  # noqa: E402
from block_sparse_attention_builder_gb300 import build as B  # noqa: E402
from block_sparse_attention_builder_gb300 import workloads as W  # noqa: E402
from tests import gpu_util as U  # noqa: E402


def _noalloc(lib, prob, inp, out, lse):
    f = lib.mxsa_attention_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 11
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return f(ctypes.byref(prob), p(inp["q"]), p(inp["k"]), p(inp["v"]), p(inp["sel"]), p(inp["bt"]), p(inp["cu"]),
             p(inp["lens"]), p(out), p(lse), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_regular_entry_points_on_two_calls():
    B.build()
    lib = mx.library()
    cases = [W.workload("tiny_decode"),
             W.custom("noalloc_small", [1, 3, 40], [700, 1300, 2100], 16, 2, 64, 4, True, "uniform", 201)]
    for w in cases:
        inp = U.device_inputs(w)
        prob = U.problem(w)
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full((w.num_q_heads, w.total_q), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, prob, inp, out, lse) == 0
        torch.cuda.synchronize()
        _, ref_out, ref_lse, _ = U.run(w, inp)
        U.assert_close_out(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), 1e-2, f"{w.spec.name} out")
        U.assert_close_lse(lse.cpu().numpy(), ref_lse.cpu().numpy(), 2e-3, f"{w.spec.name} lse")


def test_noalloc_rejects_problems_beyond_its_array():
    B.build()
    lib = mx.library()
    w = W.workload("gqa_decode")  # its workspaces need more than the fixed array holds
    prob = U.problem(w)
    ib, sb, pb = mx.workspace_size(prob)
    assert ib + sb + pb > 16 << 20
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    inp = {k: dummy for k in ("q", "k", "v", "sel", "bt", "cu", "lens")}
    assert _noalloc(lib, prob, inp, dummy, dummy) == 3  # MXSA_ERR_WORKSPACE, nothing launched
