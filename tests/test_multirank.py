"""The multi-rank path of bench.py on CPU: two gloo ranks (spawned
processes) check that every rank gets its own batch of the same workload
recipe (weak scaling, no data-path collective), that the timing reduction
takes the slowest rank, that the whole-job value counts all ranks' tokens,
and that the reference arm runs on rank 0 only."""
import importlib.util
import io
import os
import socket
import contextlib

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        w = b.load_workload("tiny_decode", rank)
        # rank-dependent batch, same shapes
        sel = torch.from_numpy(w.selected.astype(np.int64))
        lens = torch.from_numpy(w.used_kv_lens.astype(np.int64))
        gathered = [torch.zeros_like(sel) for _ in range(world)]
        dist.all_gather(gathered, sel)
        glens = [torch.zeros_like(lens) for _ in range(world)]
        dist.all_gather(glens, lens)
        # timing: rank r measured 10 + r ms over 4 steps of w.total_q tokens
        total = b.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
        value = b.whole_job_value(w.total_q, world, 4, total)
        # reference arm: rank 0 prints one line, the others nothing
        args = type("A", (), dict(workload="tiny_decode", steps=1, warmup=0))()
        buf = io.StringIO()
        printed = None
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                b.run_reference(args, rank, world)
            printed = buf.getvalue()
        out[rank] = dict(shapes=[tuple(g.shape) for g in gathered],
                         differ=not torch.equal(gathered[0], gathered[1]) or not torch.equal(glens[0], glens[1]),
                         total=total, value=value, tokens=w.total_q, printed=printed)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    r0, r1 = out[0], out[1]
    assert r0["shapes"] == r1["shapes"] and len(set(r0["shapes"])) == 1  # same per-rank work
    assert r0["differ"] and r1["differ"]  # each rank its own batch
    assert r0["total"] == r1["total"] == 11.0  # the slowest rank
    assert r0["value"] == r1["value"] == pytest.approx(r0["tokens"] * 2 * 4 / 0.011)
    assert r1["printed"] == ""  # rank 1 does no reference work


def test_single_rank_reduction_is_identity():
    b = _bench()
    assert b.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert b.whole_job_value(64, 1, 10, 2.0) == pytest.approx(64 * 10 / 0.002)
