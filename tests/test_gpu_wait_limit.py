"""A bounded on-device wait that runs out, on the GPU.

Every wait in the library's kernels gives up after a wall-clock limit, sets
MXSA_FLAG_TIMEOUT in the status word and lets the kernel return.  This test
makes one such wait run out for real: the test-only library (built beside
libmxsa.so with a 50 ms limit) has a switch that keeps one CTA of the
cooperative plan launch (index + schedule) from arriving at a grid barrier,
so every other CTA's barrier wait expires.  The launch must return (no
hang, no fault), the status word must carry MXSA_FLAG_TIMEOUT, and normal
calls in the same process -- through the test library with the switch off,
and through the regular library -- must still match the oracle.

Only the plan's grid barrier is exercised: it is integer work with no
copies or MMAs in flight, so giving up there leaves nothing to drain.
"""
import time

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

FLAG_TIMEOUT = 32


def _with_library(lib, fn):
    old = mx._lib_handle
    mx._lib_handle = lib
    try:
        return fn()
    finally:
        mx._lib_handle = old


@pytest.mark.parametrize("name,barrier", [("decode", 1), ("prefill", 2)])
def test_plan_barrier_wait_runs_out_and_the_next_calls_are_correct(name, barrier):
    B.build()
    test_lib = mx._load_library(B.TEST_LIB)
    if name == "decode":  # all-decode batch: the plan's one-barrier form
        w = W.custom("wait_decode", [1] * 40, list(range(300, 300 + 40 * 97, 97)), 16, 2, 64, 8, False,
                     "uniform", 401)
    else:  # several tokens per sequence: the general form, three barriers
        w = W.custom("wait_prefill", [5, 1, 33], [700, 1300, 2100], 16, 2, 128, 6, True, "uniform", 402)
    inp = U.device_inputs(w)
    prob = U.problem(w)

    def timed_out_plan():
        attn = mx.SparseAttention(prob, "cuda")
        assert test_lib.mxsa_test_skip_barrier_arrival(3, barrier) == 0
        try:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            attn.prepare(inp["sel"], inp["cu"], inp["lens"])
            flags = attn.status()  # synchronises
            dt = time.perf_counter() - t0
        finally:
            assert test_lib.mxsa_test_skip_barrier_arrival(-1, 0) == 0
        return flags, dt

    flags, dt = _with_library(test_lib, timed_out_plan)
    assert flags & FLAG_TIMEOUT, f"flags {flags:#x}"
    assert dt < 5.0, f"the plan launch took {dt:.2f} s"

    o_ref, l_ref = U.oracle_full(w)

    def normal_call():
        _, out, lse, _ = U.run(w, inp)
        return out, lse

    for lib in (test_lib, mx.library()):  # the switch off, then the regular library
        out, lse = _with_library(lib, normal_call)
        U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), o_ref, U.out_tol(w), f"{name} out")
        U.assert_close_lse(lse.cpu().numpy().T.reshape(-1), l_ref, 2e-3, f"{name} lse")
