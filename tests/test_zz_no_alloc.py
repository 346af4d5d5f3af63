"""The allocation-free entry point, mxsa_attention_noalloc.

Some callers may not allocate device memory themselves: plug-ins inside a
host runtime that plans every buffer up front, or hot loops that must not
risk the device-wide synchronisation of a cudaMalloc/cudaFree.  For them the
library keeps its scratch in one fixed device array.  These tests call that
entry point through the C ABI three times in a row (small, larger, small
again, so later calls run on scratch an earlier one left behind), compare
each result with the regular four-step entry points and read its status
word back with the companion call.  The file is named so that
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


def test_noalloc_matches_regular_entry_points_on_three_calls():
    """Small, larger, then small again (the last call runs on scratch a
    larger problem left behind), the last one with lse = NULL; each output
    against the four regular steps, each status word read back."""
    B.build()
    lib = mx.library()
    small = W.workload("tiny_decode")
    larger = W.custom("noalloc_small", [1, 3, 40], [700, 1300, 2100], 16, 2, 64, 4, True, "uniform", 201)
    for w, with_lse in ((small, True), (larger, True), (small, False)):
        inp = U.device_inputs(w)
        prob = U.problem(w)
        out = torch.full_like(inp["q"], float("nan"))
        lse = torch.full((w.num_q_heads, w.total_q), float("nan"), dtype=torch.float32, device="cuda")
        if with_lse:
            assert _noalloc(lib, prob, inp, out, lse) == 0
        else:
            mx.attention_noalloc(prob, inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"],
                                 out, None)
        assert mx.noalloc_read_status() == 0
        torch.cuda.synchronize()
        _, ref_out, ref_lse, _ = U.run(w, inp)
        U.assert_close_out(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), 1e-2, f"{w.spec.name} out")
        if with_lse:
            U.assert_close_lse(lse.cpu().numpy(), ref_lse.cpu().numpy(), 2e-3, f"{w.spec.name} lse")
        else:
            assert torch.isnan(lse).all()  # not written


def test_noalloc_status_reports_data_errors():
    """A repeated block and an out-of-range block in one row: the call
    succeeds, and the companion status read reports SEL_DUP and SEL_RANGE."""
    B.build()
    w = W.custom("noalloc_flags", [1, 2], [700, 900], 8, 1, 64, 4, False, "uniform", 202)
    sel = w.selected
    sel[0, 0, 1] = sel[0, 0, 0]
    sel[1, 0, 2] = 99
    inp = U.device_inputs(w)
    out = torch.empty_like(inp["q"])
    mx.attention_noalloc(U.problem(w), inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"],
                         out)
    flags = mx.noalloc_read_status()
    assert flags & 1 and flags & 2


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


def test_noalloc_first_call_during_capture_is_refused():
    """In a fresh process whose library has already run the regular steps
    (the runtime's own start-up is no call to make during a capture), the
    first noalloc call, made while the stream is being captured, returns
    MXSA_ERR_INVALID_ARG before anything runs and the capture ends cleanly;
    the same call outside the capture succeeds."""
    import os
    import subprocess
    import sys
    code = r"""
import torch
import block_sparse_attention_builder_gb300 as mx
from block_sparse_attention_builder_gb300 import workloads as W
from tests import gpu_util as U
w = W.workload("tiny_decode")
inp = U.device_inputs(w)
out = torch.empty_like(inp["q"])
prob = U.problem(w)
mx.SparseAttention(prob, "cuda")(inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"])
s = torch.cuda.Stream()
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    try:
        mx.attention_noalloc(prob, inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"],
                             out, None, stream=s)
        print("NOT REFUSED")
    except mx.MxsaError as e:
        print("REFUSED", e.status)
torch.cuda.synchronize()
mx.attention_noalloc(prob, inp["q"], inp["k"], inp["v"], inp["sel"], inp["bt"], inp["cu"], inp["lens"], out)
print("STATUS", mx.noalloc_read_status())
"""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout[-1000:], r.stderr[-2000:])
    assert "REFUSED 1" in r.stdout and "STATUS 0" in r.stdout, r.stdout
