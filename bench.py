"""Benchmark of block-sparse KV-outer attention on GB300.

One step = the whole hot path (index builder and scheduler in one launch,
KV-outer forward, combine) over one batch of a synthetic workload, inputs
resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

With no --workload (or --workload all) the line carries all five sparse
workloads, skewed_decode_shared (skewed_decode on shared prefix pages,
run through the dedup index: dedup build + scheduler + forward + combine)
and gqa_decode_nvfp4 (gqa_decode on an NVFP4 cache):
each is measured in turn (its own warm-up, timed steps, end-to-end steps and
oracle baseline) and listed under "workloads"; the line's own value,
roofline, e2e and cpu_baseline are those of skewed_decode, the largest
workload that fits one GPU.  kv_store, dense_prefill and the top-k
selection workloads are separate runs.

Timing: W untimed warm-up steps; then K steps, each bracketed by CUDA events
on the launching stream with an L2 flush (a 256 MiB write) between steps
outside the events; device time summed over the K steps; max over ranks.
Per-kernel durations come from events recorded between the calls (plan =
index + schedule in one launch, forward, combine) on the same stream.
Multi-GPU (torchrun): every rank runs its own batch of the same workload
recipe (independent sequences, no collective on the data path); value =
tokens of all ranks / max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn tokens/s, TFLOP/s and unique-KV GB/s vs roofline, 1 GB300"
L2_FLUSH_BYTES = 256 << 20
KERNELS_PER_STEP = 3  # k_plan (index + schedule) | k_fwd (decode and KV-stationary items) | k_combine
DEFAULT_WORKLOAD = "all"
# the five sparse workloads, in order; the headline is the largest one that fits one GPU
SPARSE_WORKLOADS = ("tiny_decode", "gqa_decode", "shared_prefill", "fp8_varlen", "skewed_decode")
# run with the dedup index (mxsa_build_index_dedup + mxsa_schedule: 4 launches a step)
DEDUP_WORKLOADS = ("skewed_decode_shared", "skewed_decode_shared_p64")
# the "next" rows' variants measured in the default run besides the five
EXTRA_WORKLOADS = ("skewed_decode_shared", "gqa_decode_nvfp4")
HEADLINE_WORKLOAD = "skewed_decode"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------- peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, src="fallback")


def fwd_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("fwd.cu", "fwd_decode.cuh", "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "block_sparse_attention_builder_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def fwd_phases_label(n_dec_items: int, n_kvs_items: int) -> str:
    """k_fwd and the phases its schedule uses, from the schedule header's
    item counts."""
    if n_kvs_items == 0:
        return f"k_fwd (its decode phase: {n_dec_items} items; no KV-stationary items here)"
    if n_dec_items == 0:
        return f"k_fwd (its KV-stationary phase: {n_kvs_items} items; no decode items here)"
    return f"k_fwd (decode phase: {n_dec_items} items, KV-stationary phase: {n_kvs_items} items)"


def recorded_traffic(workload: str):
    """DRAM bytes per forward launch from a committed ncu summary, if it was
    taken on the current forward-kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "k_fwd_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("fwd_source_hash") != fwd_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks: a job of independent per-rank batches
    takes as long as its slowest rank.  No-op for one rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_rank_step: int, world: int, steps: int, total_ms: float) -> float:
    """Tokens of all ranks per second, over the max-over-ranks time."""
    return tokens_per_rank_step * world * steps / (total_ms / 1e3)


# ------------------------------------------------------------- workload
def load_workload(name: str, rank: int):
    from block_sparse_attention_builder_gb300 import workloads as W
    spec = W.WORKLOADS[name]
    if rank:
        import dataclasses
        spec = dataclasses.replace(spec, seed=spec.seed + 7919 * rank)
    return W.make_workload(spec)


def workload_config(w, stats, name):
    return {"workload": name, "description": w.spec.description, "num_seqs": w.num_seqs, "total_q": w.total_q,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": 128,
            "page_size": w.page_size, "topk": w.topk, "causal": bool(w.causal), "q_dtype": w.spec.q_dtype,
            "kv_dtype": w.spec.kv_dtype, "unique_kv_blocks": stats["unique_blocks"],
            "block_visits": stats["block_visits"], "l2": "flushed between timed steps (256 MiB write); "
            "the step's unique KV also exceeds L2", "kv_cache": "resident in HBM (model state)"}


# bytes of one cached position of one kv head (K or V)
KV_ROW_BYTES = {"bf16": 256, "fp16": 256, "fp8": 128, "nvfp4": 72}


def algorithmic(w, stats):
    unique_kv_bytes = stats["unique_tokens"] * KV_ROW_BYTES[w.spec.kv_dtype] * 2
    flops = 4 * 128 * stats["visit_keys"] * (w.num_q_heads // w.num_kv_heads)
    io_bytes = (w.total_q * w.num_q_heads * 128 * 2 * 2 + w.total_q * w.num_q_heads * 4 + w.selected.nbytes
                + w.block_tables.nbytes + w.cu_seqlens_q.nbytes + w.used_kv_lens.nbytes)
    # one partial row per (row, block visit): 128 values (FP32 with FP8
    # caches, else the 16-bit q dtype) and an FP32 lse, written by the
    # forward and read back by the combine
    ps = 4 if w.spec.kv_dtype in ("fp8", "nvfp4") else 2
    partial_bytes = stats["block_visits"] * (w.num_q_heads // w.num_kv_heads) * (128 * ps + 4) * 2
    return unique_kv_bytes, flops, io_bytes, partial_bytes


# ------------------------------------------------------------ CPU oracle
def _gen_device():
    return "cuda" if torch.cuda.is_available() else "cpu"


def oracle_sample(w, target_rows: int, seed: int = 0):
    """A bounded sample of the workload for the oracle: every head of
    randomly chosen (token, kv head) pairs (all pairs when target_rows covers
    the workload), with a compact cache of the pages they reach.  The pages
    come from the seeded generator (run on the GPU when there is one, for
    speed; the bits are device-independent), never from the CUDA path."""
    import oracle
    rng = np.random.default_rng(seed)
    G = w.num_q_heads // w.num_kv_heads
    n_all = w.total_q * w.num_kv_heads
    n_pairs = max(1, min(n_all, target_rows // G))
    pairs = np.arange(n_all) if n_pairs == n_all else np.sort(rng.choice(n_all, size=n_pairs, replace=False))
    rows = (((pairs // w.num_kv_heads) * w.num_q_heads + (pairs % w.num_kv_heads) * G)[:, None]
            + np.arange(G)).reshape(-1)
    kc, vc, bt = w.compact_cache_for_rows(rows, _gen_device())
    prob = oracle.problem_for(w)
    prob.num_pages = max(1, kc.shape[0])
    return prob, w.q(), kc, vc, bt, rows


def time_oracle(w, sample, nthreads):
    import oracle
    prob, q, kc, vc, bt, rows = sample
    t0 = time.perf_counter()
    oracle.attention_rows(prob, q, kc, vc, w.selected, bt, w.cu_seqlens_q, w.used_kv_lens, rows=rows,
                          nthreads=nthreads)
    return time.perf_counter() - t0


def _sample_rows(w, nthreads, seconds):
    """Rows the oracle finishes in about `seconds` (capped at the workload)."""
    calib = oracle_sample(w, 64)
    per_row = time_oracle(w, calib, nthreads) / len(calib[-1])
    return int(max(64, min(seconds / max(per_row, 1e-9), 16384)))


def cpu_baseline(w, budget_s: float = 12.0):
    """The oracle as it stands, timed on the host cores: repeated passes over
    a bounded sample until about `budget_s` seconds of CPU work."""
    import oracle  # noqa: F401  (built by __graft_entry__.build)
    nthreads = os.cpu_count() or 1
    sample = oracle_sample(w, _sample_rows(w, nthreads, budget_s), seed=1)
    rows = len(sample[-1])
    total, passes = 0.0, 0
    while total < budget_s and passes < 50:
        total += time_oracle(w, sample, nthreads)
        passes += 1
    tok_s = rows * passes / w.num_q_heads / total
    G = w.num_q_heads // w.num_kv_heads
    whole = rows == w.total_q * w.num_q_heads
    what = "the whole workload" if whole else f"every head of {rows // G} random (token, kv-head) pairs"
    return {"value": tok_s, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{rows} (token, head) rows of {w.spec.name} ({what}), {passes} passes, {total:.1f} s "
                      f"on {nthreads} threads; tokens/s = rows / Hq / time"}


def run_reference_extra(args, world):
    """The reference arm of the store and dense workloads: the oracle's store
    of 512 tokens' K and V, or the oracle on the dense workload's last 4
    tokens, per step, on the host cores."""
    import oracle
    from block_sparse_attention_builder_gb300 import workloads as W
    if args.workload == "kv_store":
        m, hkv, ps = 512, STORE_HKV, STORE_PS
        key = W.stream_key(2000, 0)
        src = W.generate_values(m * hkv * 128, key, "bf16", "cpu").view(m, hkv, 128)
        cache = np.zeros((m // ps + 1, hkv, ps, 128), dtype=np.uint8)
        sl = np.arange(m, dtype=np.int64)

        def step():
            oracle.store(src, sl, cache, ps, "bf16", "fp8")  # K
            oracle.store(src, sl, cache, ps, "bf16", "fp8")  # V
        tokens, cores = m, 1
        metric, dtype = "kv-store tokens/s and GB/s vs HBM roofline, 1 GB300", "bf16->e4m3"
        config = {"workload": "kv_store", "tokens": STORE_TOKENS, "num_kv_heads": hkv, "page_size": ps,
                  "index_dim": STORE_IDX_DIM}
        sample = f"{m} tokens' K and V ({hkv} heads x 128, bf16 -> e4m3) per step, one thread"
    else:
        w = dense_workload(0)
        tq, hq, ps = w.total_q, w.num_q_heads, w.page_size
        rows = np.arange((tq - 4) * hq, tq * hq, dtype=np.int64)
        sel = np.arange(w.max_pages_per_seq * ps // 128, dtype=np.int32)[None, None, :].repeat(tq, 0)
        oprob = oracle.problem(1, tq, hq, w.num_kv_heads, sel.shape[2], ps, w.num_pages, w.max_pages_per_seq, True)
        qc, kc, vc = w.q(), w.k_cache(), w.v_cache()

        def step():
            oracle.attention_rows(oprob, qc, kc, vc, sel, w.block_tables, w.cu_seqlens_q, w.used_kv_lens, rows=rows)
        tokens, cores = 4, os.cpu_count() or 1
        metric, dtype = "dense-attn tokens/s and TFLOP/s vs tensor roofline, 1 GB300", "f64"
        config = {"workload": "dense_prefill", "num_q_heads": hq, "num_kv_heads": w.num_kv_heads, "page_size": ps}
        sample = f"the last 4 tokens (x {hq} heads, every key) per step"
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    total = time.perf_counter() - t0
    value = tokens * args.steps / total
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload in ("kv_store", "dense_prefill"):
        run_reference_extra(args, world)
        return
    if args.workload in SELECT_WORKLOADS:
        run_reference_select(args, world)
        return
    w = load_workload(args.workload, 0)
    nthreads = os.cpu_count() or 1
    per_step_budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    sample = oracle_sample(w, _sample_rows(w, nthreads, per_step_budget), seed=1)
    rows = len(sample[-1])
    for _ in range(args.warmup):
        time_oracle(w, sample, nthreads)
    total = 0.0
    for _ in range(args.steps):
        total += time_oracle(w, sample, nthreads)
    tokens = rows / w.num_q_heads
    value = tokens * args.steps / total
    stats = _stats(w)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, stats, args.workload),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                             "sample": f"{rows} (token, head) rows of {w.spec.name} per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _stats(w):
    from block_sparse_attention_builder_gb300 import workloads as W
    return W.selected_blocks_tokens(w)


# ---------------------------------------------------------------- main
# ----------------------------------------------------------- cache store
STORE_TOKENS, STORE_HKV, STORE_PS, STORE_IDX_DIM = 32768, 8, 128, 128


def run_store(args, rank, world, local_rank):
    """--workload kv_store: the paged-cache store (mxsa_store_kv) on a long
    prefill chunk: 32768 new tokens' K and V ([n, 8, 128] bf16) and index keys
    ([n, 1, 128] bf16) cast to e4m3 into paged caches (page 128, shuffled
    slots).  HBM-bound: value = tokens/s; roofline = bytes read + written per
    launch / event-timed launch time, against the measured copy bandwidth."""
    import block_sparse_attention_builder_gb300 as mx
    from block_sparse_attention_builder_gb300 import build as B
    from block_sparse_attention_builder_gb300 import workloads as W
    B.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    n, hkv, ps, idim = STORE_TOKENS, STORE_HKV, STORE_PS, STORE_IDX_DIM
    pages = n // ps + 8
    key = W.stream_key(2000 + rank, 0)
    k = W.generate_values(n * hkv * 128, key, "bf16", dev).view(n, hkv, 128)
    v = W.generate_values(n * hkv * 128, key + 1, "bf16", dev).view(n, hkv, 128)
    ik = W.generate_values(n * idim, key + 2, "bf16", dev).view(n, 1, idim)
    rng = np.random.default_rng(2000 + rank)
    loc_h = torch.from_numpy(rng.permutation(pages * ps)[:n].astype(np.int64))
    loc = loc_h.to(dev)
    prob = mx.make_problem(1, n, hkv, hkv, 1, ps, pages, pages, False, q_dtype=torch.bfloat16,
                           kv_dtype=torch.float8_e4m3fn)
    kc = torch.zeros(pages, hkv, ps, 128, dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    ic = torch.zeros(pages, 1, ps, idim, dtype=torch.uint8, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    bytes_read = n * (hkv * 128 * 2 * 2 + idim * 2) + n * 8
    bytes_written = n * (hkv * 128 * 2 + idim)

    def step():
        mx.store_kv(prob, loc, k, v, kc, vc, idx_k=ik, idx_cache=ic, flags=flags, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in ev), world, dev)
    ms = total_ms / args.steps
    if int(flags.item()):
        raise RuntimeError(f"store flagged {int(flags.item()):#x}")
    # end to end: this step's new rows and slots from pinned host memory, the
    # status word back
    hk, hv, hi = (t.cpu().pin_memory() for t in (k, v, ik))
    hl = loc_h.pin_memory()
    hf = torch.zeros(1, dtype=torch.int32).pin_memory()
    dk, dv, di, dl = torch.empty_like(k), torch.empty_like(v), torch.empty_like(ik), torch.empty_like(loc)
    h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hi, hl))
    e2e_ms = 0.0
    for _ in range(max(3, args.steps // 2)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for d, h in ((dk, hk), (dv, hv), (di, hi), (dl, hl)):
            d.copy_(h, non_blocking=True)
        mx.store_kv(prob, dl, dk, dv, kc, vc, idx_k=di, idx_cache=ic, flags=flags, stream=stream)
        hf.copy_(flags, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= max(3, args.steps // 2)
    peaks = measured_peaks()
    gbs = (bytes_read + bytes_written) / (ms / 1e3) / 1e9
    line = {
        "metric": "kv-store tokens/s and GB/s vs HBM roofline, 1 GB300", "value": n * world / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
        "data": "synthetic (seeded counter-based N(0,1) values, shuffled slots)",
        "config": {"workload": "kv_store", "description": "32768 new tokens, K/V [n,8,128] + index keys [n,1,128] "
                   "bf16 -> e4m3 paged caches, page 128, shuffled slots", "tokens": n, "num_kv_heads": hkv,
                   "page_size": ps, "index_dim": idim, "l2": "flushed between timed steps (256 MiB write)"},
        "bytes": {"read": bytes_read, "written": bytes_written},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "k_store",
                     "peak_source": peaks["src"]},
        "e2e": {"value": n / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps, "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = store_oracle_baseline(k[:512].cpu(), ps, 10.0)
    if rank == 0:
        print(json.dumps(line), flush=True)


def store_oracle_baseline(src, ps, budget_s):
    """The oracle's store (single-threaded) of the K and V rows `src`
    ([m, Hkv, 128] bf16, CPU) into an e4m3 cache, repeated for about
    `budget_s` seconds."""
    import oracle
    m, hkv = int(src.shape[0]), int(src.shape[1])
    cache = np.zeros((m // ps + 1, hkv, ps, 128), dtype=np.uint8)
    sl = np.arange(m, dtype=np.int64)
    t0 = time.time()
    reps = 0
    while time.time() - t0 < budget_s or reps == 0:
        oracle.store(src, sl, cache, ps, "bf16", "fp8")
        oracle.store(src, sl, cache, ps, "bf16", "fp8")
        reps += 1
    dt = time.time() - t0
    return {"value": m * reps / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{m} tokens' K and V ({hkv} heads x 128, bf16 -> e4m3), {reps} passes, "
                      f"{dt:.1f} s on one thread (the oracle's store is single-threaded)"}


# ------------------------------------------------------------ dense path
def run_dense(args, rank, world, local_rank):
    """--workload dense_prefill: the dense path (mxsa_dense_fwd: every key,
    no partials) on the shared-prefill shape (1 sequence, 4096 new tokens on
    L = 36864, Hq 16 / Hkv 1, page 128, causal).  value = tokens/s; roofline
    = causal FLOPs (4 * 128 per query head and visible key) per launch / the
    event-timed launch, against the measured BF16 dense peak."""
    import block_sparse_attention_builder_gb300 as mx
    from block_sparse_attention_builder_gb300 import build as B
    from block_sparse_attention_builder_gb300 import workloads as W
    B.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    tq, L, hq, hkv, ps = 4096, 36864, 16, 1, 128
    w = dense_workload(rank)
    q, k, v = w.q(dev), w.k_cache(dev), w.v_cache(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cu = torch.from_numpy(w.cu_seqlens_q).to(dev)
    lens = torch.from_numpy(w.used_kv_lens).to(dev)
    prob = mx.make_problem(1, tq, hq, hkv, 1, ps, w.num_pages, w.max_pages_per_seq, True)
    out = torch.empty_like(q)
    lse = torch.empty(hq, tq, dtype=torch.float32, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    keys = tq * (L - tq) + tq * (tq + 1) // 2  # visible keys summed over the tokens
    flops = 4.0 * 128 * hq * keys

    def step():
        mx.dense_fwd(prob, q, k, v, bt, cu, lens, out, lse, flags=flags, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in ev), world, dev)
    ms = total_ms / args.steps
    if int(flags.item()):
        raise RuntimeError(f"dense path flagged {int(flags.item()):#x}")
    # end to end: q from pinned host memory, out and lse back to pinned host
    hq_h = q.cpu().pin_memory()
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    dq = torch.empty_like(q)
    e2e_ms, reps = 0.0, max(3, args.steps // 2)
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dq.copy_(hq_h, non_blocking=True)
        mx.dense_fwd(prob, dq, k, v, bt, cu, lens, out, lse, flags=flags, stream=stream)
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= reps
    peaks = measured_peaks()
    tf = flops / (ms / 1e3) / 1e12
    line = {
        "metric": "dense-attn tokens/s and TFLOP/s vs tensor roofline, 1 GB300", "value": tq * world / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based N(0,1) values)",
        "config": {"workload": "dense_prefill", "description": "1 seq, Tq=4096 on L=36864, Hq16/Hkv1, ps128, causal, "
                   "every key (no selection)", "num_q_heads": hq, "num_kv_heads": hkv, "page_size": ps,
                   "l2": "flushed between timed steps (256 MiB write)"},
        "flops": flops,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tf / peaks["bf16_tflops"], "traffic": None, "kernel": "k_dense",
                     "peak_source": peaks["src"]},
        "e2e": {"value": tq / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": q.numel() * q.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size() + lse.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps, "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = dense_oracle_baseline(w, 10.0)
    if rank == 0:
        print(json.dumps(line), flush=True)


def dense_workload(rank):
    """The dense path's workload: 1 sequence, 4096 new tokens on L = 36864,
    Hq 16 / Hkv 1, page 128, causal, every block."""
    from block_sparse_attention_builder_gb300 import workloads as W
    return W.custom("dense_prefill", [4096], [36864], 16, 1, 128, 1, True, "uniform", 3000 + rank)


def dense_oracle_baseline(w, budget_s):
    """The oracle on the dense workload's last 4 tokens (the longest rows,
    every key), repeated for about `budget_s` seconds."""
    import oracle
    tq, hq, hkv, ps = w.total_q, w.num_q_heads, w.num_kv_heads, w.page_size
    L = int(w.used_kv_lens[0])
    rows = np.arange((tq - 4) * hq, tq * hq, dtype=np.int64)
    sel = np.arange(w.max_pages_per_seq * ps // 128, dtype=np.int32)[None, None, :].repeat(tq, 0)
    oprob = oracle.problem(1, tq, hq, hkv, sel.shape[2], ps, w.num_pages, w.max_pages_per_seq, True)
    qc, kc, vc = w.q(), w.k_cache(), w.v_cache()
    t0 = time.time()
    reps = 0
    while time.time() - t0 < budget_s or reps == 0:
        oracle.attention_rows(oprob, qc, kc, vc, sel, w.block_tables, w.cu_seqlens_q, w.used_kv_lens, rows=rows)
        reps += 1
    dt = time.time() - t0
    return {"value": 4 * reps / dt, "unit": "tokens/s", "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": f"the last 4 tokens (x {hq} heads, ~{L} keys each), {reps} passes, "
                      f"{dt:.1f} s; tokens/s = tokens / time"}


def run_sparse(name, args, rank, world, local_rank, cpu_budget_s):
    """One sparse workload: W warm-up steps, K timed steps (device time per
    kernel from events on the launching stream, L2 flushed between steps),
    then the same steps end to end through the public API with host buffers.
    Returns the workload's JSON entry (rank 0) or None."""
    import block_sparse_attention_builder_gb300 as mx
    dev = torch.device("cuda", local_rank)
    from block_sparse_attention_builder_gb300 import workloads as W
    dedup = name in DEDUP_WORKLOADS if args.index == "auto" else args.index == "dedup"
    w = load_workload(name, rank)
    stats = _stats(w)
    if dedup:  # a shared block is loaded once for every sequence that holds it
        phys = W.physical_blocks_tokens(w)
        stats["unique_blocks_per_sequence"] = stats["unique_blocks"]
        stats["unique_blocks"], stats["unique_tokens"] = phys["unique_blocks"], phys["unique_tokens"]
    unique_kv_bytes, flops, io_bytes, partial_bytes = algorithmic(w, stats)
    log(f"[bench] {name}: {stats}")

    # inputs resident in HBM
    q, k, v = w.q(dev), w.k_cache(dev), w.v_cache(dev)
    sel = torch.from_numpy(w.selected).to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cu = torch.from_numpy(w.cu_seqlens_q).to(dev)
    lens = torch.from_numpy(w.used_kv_lens).to(dev)
    prob = mx.make_problem(w.num_seqs, w.total_q, w.num_q_heads, w.num_kv_heads, w.topk, w.page_size,
                           w.num_pages, w.max_pages_per_seq, w.causal, 0.0, q.dtype,
                           "nvfp4" if w.spec.kv_dtype == "nvfp4" else k.dtype)
    attn = mx.SparseAttention(prob, dev, dedup=dedup)
    out = torch.empty_like(q)
    lse = torch.empty(w.num_q_heads, w.total_q, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        if dedup:  # the index keyed by physical block, then the scheduler
            mx.build_index_dedup(prob, sel, cu, lens, bt, attn.ws.index, attn.dedup_ws, stream)
            mx.schedule(prob, attn.ws.index, attn.ws.sched, 0, stream)
        elif args.plan == "separate":  # the two steps as their own launches (k_index, k_schedule)
            mx.build_index(prob, sel, cu, lens, attn.ws.index, stream)
            mx.schedule(prob, attn.ws.index, attn.ws.sched, 0, stream)
        else:
            mx.plan(prob, sel, cu, lens, attn.ws.index, attn.ws.sched, 0, stream)  # index + schedule, one launch
        if ev:
            ev[1].record(stream)
        mx.kvouter_fwd(prob, q, k, v, bt, attn.ws.index, attn.ws.sched, attn.ws.partial, 0, stream)
        if ev:
            ev[2].record(stream)
        mx.combine(prob, attn.ws.index, attn.ws.partial, out, lse, stream)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = mx.read_status(attn.ws.index, stream)
    if flags:
        raise RuntimeError(f"{name}: device status flags {flags:#x} after warm-up")
    # which of the forward's phases this schedule uses (the schedule
    # header's item counts: KV-stationary items, decode items)
    hdr_off = mx.sched_layout(prob).header
    sch_hdr = attn.ws.sched[hdr_off:hdr_off + 64].view(torch.int32).cpu()
    n_kvs_items, n_dec_items = int(sch_hdr[0]), int(sch_hdr[5])

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for i in range(args.steps):
        flush.zero_()
        step(events[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    per = np.array([[events[i][j].elapsed_time(events[i][j + 1]) for j in range(3)] for i in range(args.steps)])
    step_ms = per.sum(axis=1)
    total_ms = max_over_ranks(float(step_ms.sum()), world, dev)
    ms_per_step = total_ms / args.steps
    tokens_per_step = w.total_q
    value = whole_job_value(tokens_per_step, world, args.steps, total_ms)
    fwd_ms = float(per[:, 1].mean())
    peaks = measured_peaks()

    # ---------------------------------------------------------- e2e (public API, host buffers)
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_bt = pin(q), pin(bt)
    # the plan's small inputs live in one pinned staging buffer (and one
    # device buffer), so they cross in one copy: cu_seqlens_q (int64) first,
    # then the selections and the lengths, each at a 256-byte boundary
    small = [cu, sel, lens]
    offs, off = [], 0
    for t_ in small:
        offs.append(off)
        off += (t_.numel() * t_.element_size() + 255) // 256 * 256
    h_small = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_small = torch.empty(off, dtype=torch.uint8, device=dev)

    def view(buf, i):
        t_ = small[i]
        n = t_.numel() * t_.element_size()
        return buf[offs[i]:offs[i] + n].view(t_.dtype).view(t_.shape)

    h_cu, h_sel, h_lens = (view(h_small, i) for i in range(3))
    d_cu, d_sel, d_lens = (view(d_small, i) for i in range(3))
    for h_, t_ in ((h_cu, cu), (h_sel, sel), (h_lens, lens)):
        h_.copy_(t_.cpu())
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d_q, d_bt = torch.empty_like(q), torch.empty_like(bt)
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_sel, h_bt, h_cu, h_lens))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

    # The user's call sequence: the plan's inputs (selections, lengths) go
    # first and the plan runs while q and the block tables copy on a second
    # stream; the combine writes out and lse straight into the pinned host
    # buffers (no device-to-host copy; the bytes cross the host link).
    e2e_stream, side = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = torch.cuda.Event()

    def e2e_step():
        side.wait_stream(e2e_stream)  # the previous step's forward is done with d_q / d_bt
        with torch.cuda.stream(side):
            d_q.copy_(h_q, non_blocking=True)
            d_bt.copy_(h_bt, non_blocking=True)
            ev_in.record(side)
        with torch.cuda.stream(e2e_stream):
            d_small.copy_(h_small, non_blocking=True)
        if dedup:  # the dedup index reads the block tables too
            e2e_stream.wait_event(ev_in)
        attn.prepare(d_sel, d_cu, d_lens, stream=e2e_stream, block_tables=d_bt)
        e2e_stream.wait_event(ev_in)
        attn.attend(d_q, k, v, d_bt, out=h_out, lse=h_lse, stream=e2e_stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = 0.0
    for _ in range(args.steps):
        flush.zero_()
        e2e_stream.wait_stream(torch.cuda.current_stream(dev))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(e2e_stream)
        e2e_step()
        e1.record(e2e_stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = whole_job_value(tokens_per_step, world, args.steps, e2e_ms)
    assert torch.equal(h_out.to(dev), out)
    del q, k, v, attn, flush, d_q, d_small
    torch.cuda.empty_cache()
    if rank != 0:
        return None

    kv_gbs = unique_kv_bytes / (ms_per_step / 1e3) / 1e9
    tflops = flops / (ms_per_step / 1e3) / 1e12
    fwd_gbs = unique_kv_bytes / (fwd_ms / 1e3) / 1e9
    fwd_tflops = flops / (fwd_ms / 1e3) / 1e12
    bound = "hbm" if "decode" in w.spec.name else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": fwd_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": fwd_gbs / peaks["hbm_gbs"], "traffic": recorded_traffic(name),
                "kernel": fwd_phases_label(n_dec_items, n_kvs_items),
                "algorithmic_bytes_per_launch": unique_kv_bytes, "peak_source": peaks["src"] + " copy bandwidth"}
    else:
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": fwd_tflops, "peak": pk, "unit": "TFLOP/s",
                "frac": fwd_tflops / pk, "traffic": recorded_traffic(name),
                "kernel": fwd_phases_label(n_dec_items, n_kvs_items),
                "algorithmic_flops_per_launch": flops, "peak_source": peaks["src"] + " bf16 burst"}
    step_roof = {"hbm_frac": kv_gbs / peaks["hbm_gbs"], "tensor_frac": tflops / peaks["bf16_tflops"]}
    entry = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"fp8": "fp8-e4m3 kv, bf16 q", "nvfp4": "nvfp4 kv (e2m1 + e4m3 scale per 16), bf16 q"}.get(
            w.spec.kv_dtype, w.spec.kv_dtype),
        "data": "synthetic (seeded counter-based N(0,1) values; selections per the workload recipe)",
        "config": workload_config(w, stats, name),
        "tflops": tflops, "unique_kv_gbs": kv_gbs, "step_roofline": step_roof,
        "kernel_ms": {("dedup index + schedule" if dedup else "plan (index + schedule)"): float(per[:, 0].mean()),
                      "fwd": fwd_ms,
                      "combine": float(per[:, 2].mean())},
        "fwd_unique_kv_gbs": fwd_gbs, "fwd_tflops": fwd_tflops,
        "bytes": {"unique_kv": unique_kv_bytes, "io": io_bytes, "partials_overhead": partial_bytes},
        "flops": flops,
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "note": "every step: selections, cu_seqlens_q, used_kv_lens copied H2D in one copy from "
                        "one pinned staging buffer, then the plan while q and block tables copy on a second "
                        "stream; the combine writes out + lse into pinned host memory directly (counted as "
                        "D2H bytes); the KV cache is resident model state"},
        "gpu_launches": (KERNELS_PER_STEP + (dedup or args.plan == "separate")) * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline(w, cpu_budget_s)
    return entry


# --------------------------------------------------------- top-k selection
SELECT_WORKLOADS = {"select_decode": ("gqa_decode", 64), "select_prefill": ("shared_prefill", 128)}


def select_visible_keys(w):
    """Sum over (token, kv head) rows of the positions their blocks are
    scored over (p < L, and p <= pos(t) when causal): the dot products."""
    n = 0
    for s in range(w.num_seqs):
        L = int(w.used_kv_lens[s])
        t0, t1 = int(w.cu_seqlens_q[s]), int(w.cu_seqlens_q[s + 1])
        for i in range(t1 - t0):
            n += min(L, L - (t1 - t0) + i + 1) if w.causal else L
    return n * w.num_kv_heads


def select_oracle_step(w, dim):
    """One pass of the oracle's selection over 32 rows of a few sequences (a
    compact copy of their index pages): (step callable, rows, description)."""
    import oracle
    rng = np.random.default_rng(1)
    seqs = sorted(rng.choice(w.num_seqs, size=min(4, w.num_seqs), replace=False).tolist())
    pages = sorted({int(p) for s in seqs for p in w.block_tables[s] if p >= 0})
    remap = {p: i for i, p in enumerate(pages)}
    bt = np.full_like(w.block_tables, -1)
    for s in seqs:
        for j, p in enumerate(w.block_tables[s]):
            if p >= 0:
                bt[s, j] = remap[int(p)]
    ikc = w.idx_cache_pages(dim, np.array(pages), _gen_device())
    iq = w.idx_q(dim)
    prob = oracle.problem_for(w)
    prob.num_pages = len(pages)
    rows = np.concatenate([np.arange(w.cu_seqlens_q[s] * w.num_kv_heads, w.cu_seqlens_q[s + 1] * w.num_kv_heads)
                           for s in seqs])
    rows = np.sort(rng.choice(rows, size=min(len(rows), 32), replace=False))
    nthreads = os.cpu_count() or 1

    def step():
        oracle.select_blocks(prob, dim, iq, ikc, bt, w.cu_seqlens_q, w.used_kv_lens, rows=rows, nthreads=nthreads)
    return step, len(rows), f"{len(rows)} (token, kv head) rows of sequences {seqs} on {nthreads} threads"


def select_oracle_sample(w, dim, budget_s):
    """The oracle's selection sample, repeated for about budget_s seconds."""
    step, nrows, what = select_oracle_step(w, dim)
    t0, reps = time.time(), 0
    while time.time() - t0 < budget_s or reps == 0:
        step()
        reps += 1
    dt = time.time() - t0
    return {"value": nrows * reps / w.num_kv_heads / dt, "unit": "tokens/s", "cores": os.cpu_count() or 1,
            "kind": "oracle", "sample": f"{what}, {reps} passes, {dt:.1f} s; tokens/s = rows / Hkv / time"}


def run_reference_select(args, world):
    """The reference arm of the selection workloads: the oracle's selection
    of 32 rows per step on the host cores."""
    base, dim = SELECT_WORKLOADS[args.workload]
    w = load_workload(base, 0)
    step, nrows, what = select_oracle_step(w, dim)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    total = time.perf_counter() - t0
    value = nrows / w.num_kv_heads * args.steps / total
    line = {"impl": "reference", "metric": "top-k block selection tokens/s vs roofline, 1 GB300", "value": value,
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 scores", "data": "synthetic",
            "config": {"workload": args.workload, "shape_of": base, "index_dim": dim},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count() or 1, "kind": "oracle",
                             "sample": what + " per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_select(args, rank, world, local_rank):
    """--workload select_decode | select_prefill: the top-k block selection
    (mxsa_select_blocks) on the gqa_decode shape with 64-dim index keys, or
    the shared_prefill shape with 128-dim index keys (bf16, one index head
    per kv head).  value = tokens/s.  select_decode is HBM-bound (the index
    cache is read once); select_prefill is bound by the CUDA-core FP32 FMAs
    the exact scores take (alu)."""
    import block_sparse_attention_builder_gb300 as mx
    from block_sparse_attention_builder_gb300 import build as B
    B.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    base, dim = SELECT_WORKLOADS[args.workload]
    w = load_workload(base, rank)
    iq, ik = w.idx_q(dim, dev), w.idx_cache(dim, dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cu = torch.from_numpy(w.cu_seqlens_q).to(dev)
    lens = torch.from_numpy(w.used_kv_lens).to(dev)
    prob = mx.make_problem(w.num_seqs, w.total_q, w.num_q_heads, w.num_kv_heads, w.topk, w.page_size, w.num_pages,
                           w.max_pages_per_seq, w.causal, 0.0, torch.bfloat16, torch.bfloat16)
    sel = torch.empty(w.total_q, w.num_kv_heads, w.topk, dtype=torch.int32, device=dev)
    ws = torch.empty(mx.select_workspace_size(prob, dim), dtype=torch.uint8, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        mx.select_blocks(prob, iq, ik, bt, cu, lens, sel=sel, score_ws=ws, flags=flags, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in ev), world, dev)
    ms = total_ms / args.steps
    if int(flags.item()):
        raise RuntimeError(f"selection flagged {int(flags.item()):#x}")
    # end to end: the index queries from pinned host memory, the selections back
    h_iq = iq.cpu().pin_memory()
    h_sel = torch.empty(sel.shape, dtype=sel.dtype).pin_memory()
    d_iq = torch.empty_like(iq)
    e2e_ms, reps = 0.0, max(3, args.steps // 2)
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        d_iq.copy_(h_iq, non_blocking=True)
        mx.select_blocks(prob, d_iq, ik, bt, cu, lens, sel=sel, score_ws=ws, flags=flags, stream=stream)
        h_sel.copy_(sel, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= reps
    peaks = measured_peaks()
    visible = select_visible_keys(w)
    cache_bytes = sum(int(w.used_kv_lens[s]) for s in range(w.num_seqs)) * w.num_kv_heads * dim * 2
    nbm = (w.max_pages_per_seq * w.page_size + 127) // 128
    io_bytes = iq.numel() * 2 + sel.numel() * 4 + 2 * w.total_q * w.num_kv_heads * nbm * 4
    if args.workload == "select_decode":
        gbs = (cache_bytes + io_bytes) / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": "k_select_score + k_select_topk",
                "algorithmic_bytes_per_launch": cache_bytes + io_bytes,
                "peak_source": peaks["src"] + " copy bandwidth"}
    else:
        fl = 2.0 * visible * dim
        alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x FP32 lanes x 2 FLOP per FMA x max SM clock
        tf = fl / (ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": tf, "peak": alu_peak, "unit": "TFLOP/s", "frac": tf / alu_peak,
                "traffic": None, "kernel": "k_select_score + k_select_topk", "algorithmic_flops_per_launch": fl,
                "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz (FP32 FMA on CUDA cores)"}
    line = {
        "metric": "top-k block selection tokens/s vs roofline, 1 GB300", "value": w.total_q * world / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 scores",
        "data": "synthetic (seeded counter-based N(0,1) index queries and keys)",
        "config": {"workload": args.workload, "shape_of": base, "index_dim": dim, "num_seqs": w.num_seqs,
                   "total_q": w.total_q, "num_kv_heads": w.num_kv_heads, "topk": w.topk, "page_size": w.page_size,
                   "causal": bool(w.causal), "dot_products": visible,
                   "l2": "flushed between timed steps (256 MiB write)"},
        "bytes": {"index_cache": cache_bytes, "io": io_bytes}, "roofline": roof,
        "e2e": {"value": w.total_q / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": iq.numel() * 2,
                "d2h_bytes_per_step": sel.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps, "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = select_oracle_sample(w, dim, 8.0)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="'all' (default): the five sparse workloads, the dedup one and the NVFP4 one in one line, headline "
                         "skewed_decode; "
                         "or one of " + ", ".join(list(SPARSE_WORKLOADS) + list(DEDUP_WORKLOADS) +
                                                  ["gqa_decode_nvfp4", "gqa_decode_p16"] +
                                                  ["kv_store", "dense_prefill"] +
                                                  list(SELECT_WORKLOADS)))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--plan", default="fused", choices=["fused", "separate"],
                    help="index + schedule in one launch (mxsa_plan, default) or as mxsa_build_index then "
                         "mxsa_schedule")
    ap.add_argument("--index", default="auto", choices=["auto", "plain", "dedup"],
                    help="the index a sparse workload runs on: auto = dedup for " + ", ".join(DEDUP_WORKLOADS) +
                         ", plain for the others")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "mine" else "gloo")

    if args.impl == "reference":
        if args.workload == "all":
            args.workload = HEADLINE_WORKLOAD
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if args.workload in ("kv_store", "dense_prefill") or args.workload in SELECT_WORKLOADS:
        run = {"kv_store": run_store, "dense_prefill": run_dense}.get(args.workload, run_select)
        run(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    from block_sparse_attention_builder_gb300 import build as B
    B.build()
    torch.cuda.set_device(local_rank)
    if args.workload == "all":
        names, headline = list(SPARSE_WORKLOADS) + list(EXTRA_WORKLOADS), HEADLINE_WORKLOAD
    else:
        names, headline = [args.workload], args.workload
    entries = {}
    for name in names:
        entries[name] = run_sparse(name, args, rank, world, local_rank, 12.0 if name == headline else 6.0)
    if rank == 0:
        line = dict(entries[headline])
        if len(names) > 1:
            line["headline"] = (f"{headline}: the largest single-GPU workload; every workload's own numbers "
                                f"(value, roofline, e2e, cpu_baseline, clocks) are under 'workloads'")
            line["workloads"] = entries
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
