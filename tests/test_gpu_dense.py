"""GPU parity of the dense path (mxsa_dense_fwd: every key of each sequence,
the all-blocks-selected case computed without partials) with the oracle's
attention on a selection of every block (the oracle's all-selected case is
pinned to torch SDPA in tests/test_oracle_pins.py)."""
import math

import numpy as np
import pytest
import torch

import block_sparse_attention_builder_gb300 as mx
import oracle
from block_sparse_attention_builder_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _dense_case(name, tq, lens, hq, hkv, ps, causal, seed, q_dtype="bf16"):
    topk = max(1, max(math.ceil(L / 128) for L in lens))
    return W.custom(name, tq, lens, hq, hkv, ps, topk, causal, "all", seed, q_dtype=q_dtype, kv_dtype=q_dtype)


CASES = {
    "prefill_g16": _dense_case("dense_g16", [130], [700], 16, 1, 128, True, 201),
    "gqa_g8_varlen": _dense_case("dense_g8", [1, 37, 5], [300, 900, 129], 16, 2, 64, True, 202),
    "mha_g1_fp16": _dense_case("dense_g1", [200], [600], 4, 4, 128, False, 203, q_dtype="fp16"),
    "g3_causal": _dense_case("dense_g3", [50, 3], [400, 64], 12, 4, 64, True, 204),
    "g128": _dense_case("dense_g128", [3, 1], [500, 130], 128, 1, 128, True, 205),
    "empty_rows": _dense_case("dense_empty", [0, 2, 3], [100, 0, 300], 8, 1, 64, False, 206),
    # 1024 sequences (the most the kernel's shared-memory table holds),
    # some without tokens, some shorter than their new tokens
    "seqs_1024": _dense_case("dense_1024", [1, 2, 0, 3] * 256,
                             [int(x) for x in np.random.default_rng(207).integers(2, 400, 1024)], 8, 1, 64, True,
                             207),
}


@pytest.mark.parametrize("name", list(CASES))
def test_dense_matches_oracle(name):
    w = CASES[name]
    inp = U.device_inputs(w)
    prob = U.problem(w)
    out = torch.full_like(inp["q"], float("nan"))
    lse = torch.full((w.num_q_heads, w.total_q), float("nan"), dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx.dense_fwd(prob, inp["q"], inp["k"], inp["v"], inp["bt"], inp["cu"], inp["lens"], out, lse, flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    o_ref, l_ref = oracle.attention_rows(oracle.problem_for(w), w.q(), w.k_cache(), w.v_cache(), w.selected,
                                         w.block_tables, w.cu_seqlens_q, w.used_kv_lens)
    o_gpu = out.float().cpu().numpy().reshape(-1, 128)
    l_gpu = lse.cpu().numpy().T.reshape(-1)  # [Hq, Tq] -> rows t * Hq + h
    U.assert_close_out(o_gpu, o_ref, U.out_tol(w), f"{name} out")
    U.assert_close_lse(l_gpu, l_ref, 2e-3, f"{name} lse")


def test_dense_equals_the_sparse_path_with_every_block_selected():
    w = CASES["gqa_g8_varlen"]
    attn, out_s, lse_s, inp = U.run(w)
    out = torch.empty_like(inp["q"])
    lse = torch.empty(w.num_q_heads, w.total_q, dtype=torch.float32, device="cuda")
    mx.dense_fwd(U.problem(w), inp["q"], inp["k"], inp["v"], inp["bt"], inp["cu"], inp["lens"], out, lse)
    torch.cuda.synchronize()
    U.assert_close_out(out.float().cpu().numpy().reshape(-1, 128), out_s.float().cpu().numpy().reshape(-1, 128),
                       U.out_tol(w), "dense vs sparse out")
    U.assert_close_lse(lse.cpu().numpy().reshape(-1), lse_s.cpu().numpy().reshape(-1), 2e-3, "dense vs sparse lse")
