"""Benchmark of the hybrid sparse MQA attention step on GB300.

One step = one call of the attention step over one batch of the workload
(key-slot resolution, gather, QK^T, sink softmax, PV, split merge, write).
Default workload: C4 top-512 decode, batch 32, H=64, D=512 bf16, context
65536 (16384 compressed rows per request) + SWA window 128.

`--workload kv_store_prefill` (or kv_store_decode) measures the cache write
that precedes the step instead: one step = one dsv4_kv_store call packing and
storing a batch of new key rows.  `--workload topk_1m` (or topk_c4_decode)
measures the top-k selection that makes the C4 index lists: one step = one
dsv4_topk call over a batch of indexer score rows.

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the workload
(requests are independent; there is no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is used.

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "query-tokens/s and achieved HBM GB/s (% roofline) for C4 top-512 sparse MQA decode"
DEFAULT_WORKLOAD = "c4_decode"
STORE_METRIC = "KV rows stored/s and achieved HBM GB/s (% roofline) for the FP8 pack-and-store cache write"
TOPK_METRIC = "query-tokens/s (rows selected) and achieved HBM GB/s (% roofline) for top-k index selection"
NOMINAL_HBM_GBS = 7900.0      # the part's nominal HBM3e rate, reported beside the measured peak


# ---------------------------------------------------------------- helpers
def slowest_ms(ms, world, device):
    """The job's time for a per-rank time `ms`: the maximum over the ranks of
    the process group (every rank's replica has to finish)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tokens_per_s(tokens_per_rank_step, world, sec_per_step):
    """Whole-job throughput: every rank processes its own batch each step."""
    return world * tokens_per_rank_step / sec_per_step


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d.get("hbm_gbs"), bf16_tflops=d.get("bf16_tflops"),
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


ATTN_SOURCES = ("hybrid_sparse_mqa_gb300/csrc/dsv4_attn.cu", "hybrid_sparse_mqa_gb300/csrc/dsv4_device.cuh")
STORE_SOURCES = ("hybrid_sparse_mqa_gb300/csrc/dsv4_kv_store.cu",)
TOPK_SOURCES = ("hybrid_sparse_mqa_gb300/csrc/dsv4_topk.cu",)


def kernel_source_hash(sources=ATTN_SOURCES):
    """Hash of a kernel's sources' code: comments and whitespace do not
    count, so a stored ncu figure stays valid until the code itself changes."""
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch of the workload's main kernel from the committed
    ncu summary, if it was taken on the current kernel source; else None."""
    if is_store_workload(workload):
        name, sources = "dsv4_kv_store_kernel_traffic.json", STORE_SOURCES
    elif is_topk_workload(workload):
        name, sources = "dsv4_topk_kernel_traffic.json", TOPK_SOURCES
    else:
        name, sources = "dsv4_attn_kernel_traffic.json", ATTN_SOURCES
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- oracle timing
_ORACLE = {}


def _oracle_init(inp):
    """Pool worker set-up: the inputs arrive as shared CPU tensors (BLAS runs
    one thread per process: the spawning parent set that in the environment
    the worker inherits)."""
    sys.path.insert(0, ROOT)
    from oracle import dsv4_oracle as O
    _ORACLE["O"] = O
    _ORACLE["kw"] = inp.oracle_kwargs()
    O.dsv4_attention(**_ORACLE["kw"], tokens=[0])


def _oracle_tokens(tokens):
    _ORACLE["O"].dsv4_attention(**_ORACLE["kw"], tokens=list(tokens))
    return len(tokens)


def oracle_pool(inp_cpu, workers):
    """A pool of `workers` spawned processes, each holding the workload's
    inputs (shared CPU tensors) and running the oracle with one BLAS thread."""
    import multiprocessing as mp
    import torch  # noqa: F401  (registers the shared-memory pickling of CPU tensors)
    for name in ("q", "seq_lens", "swa_pool", "swa_page_table", "extra_pool", "extra_page_table", "topk_idx",
                 "sink", "cu_seqlens_q", "req_pool_indices"):
        x = getattr(inp_cpu, name, None)
        if x is not None:
            x.share_memory_()
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in saved:
        os.environ[v] = "1"
    try:
        pool = mp.get_context("spawn").Pool(workers, initializer=_oracle_init, initargs=(inp_cpu,))
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    pool.map(_oracle_tokens, [[0]] * workers, chunksize=1)      # every worker is up
    return pool


def oracle_throughput(inp_cpu, workers, seconds, per_task=4):
    """Query tokens per second of the float64 oracle on this host: `workers`
    processes (one BLAS thread each), tasks of `per_task` consecutive tokens,
    best of three runs of about `seconds` each."""
    T = inp_cpu.T
    with oracle_pool(inp_cpu, workers) as pool:
        probe = [[(k * per_task + i) % T for i in range(per_task)] for k in range(workers)]
        t0 = time.perf_counter()
        pool.map(_oracle_tokens, probe, chunksize=1)
        per_round = max(time.perf_counter() - t0, 1e-4)
        rounds = max(1, int(seconds / per_round))
        tasks = [[(k * per_task + i) % T for i in range(per_task)] for k in range(rounds * workers)]
        best = 0.0
        for _ in range(3):
            t0 = time.perf_counter()
            done = sum(pool.map(_oracle_tokens, tasks, chunksize=1))
            best = max(best, done / (time.perf_counter() - t0))
    return best, rounds * workers * per_task


def rotating_sets(make, first_bytes, requested, l2):
    """Input sets for the timed rotation: `requested` if given (> 0), else
    at least 12 and enough that one rotation touches four times the L2
    (at most 512).  `make(r)` builds set r; `first_bytes(set)` is a call's
    algorithmic bytes."""
    first = make(0)
    if requested > 0:
        n = requested
    else:
        n = max(12, min(512, math.ceil(4 * l2 / max(1, first_bytes(first)))))
    return [first] + [make(r) for r in range(1, n)]


def capture_steps(step, R, steps, stream):
    """CUDA graphs that together replay `steps` calls, call k on input set
    k % R.  A short run is one graph (no graph boundary inside the timed
    region); a long one is a graph of whole rotations (about 256 calls)
    replayed as often as it fits, plus a graph of the remainder.  Returns
    the replay plan [(graph, times), ...] and (graph, calls) for warming the
    clocks."""
    import torch

    def cap(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                step(k, torch.cuda.current_stream())
        return g

    if steps <= 512:
        g = cap(steps)
        return [(g, 1)], (g, steps)
    block = R * max(1, 256 // R)
    full, rem = divmod(steps, block)
    g = cap(block)
    plan = [(g, full)]
    if rem:
        plan.append((cap(rem), 1))
    return plan, (g, block)


def capture_lead(step, R, stream):
    """A one-call graph on the last input set, run right before the timed
    region so that the switch from the spin kernel to the measured kernel
    (its shared-memory configuration, its first launch) happens outside it;
    the first timed call (set 0) was last touched a whole rotation earlier."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(R - 1, torch.cuda.current_stream())
    return g


def replay(plan):
    for g, times in plan:
        for _ in range(times):
            g.replay()


def hold_stream(stream, lead=None, cycles=2_000_000):
    """Keep the launch stream busy for a fixed number of GPU cycles (about
    1 ms; the spin reads nothing and waits on nothing) so that the host has
    enqueued the timed graph replays before the first of them starts: the
    timed region then holds the kernels back to back, not the host's launch
    latency.  `lead` (a graph) runs after the spin, before the timed region."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(cycles)
        if lead is not None:
            lead.replay()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        t0, t1 = (self.marks + [0, 0])[:2] if len(self.marks) >= 2 else (0, 1e30)
        inside = [l for (t, l) in self.lines if t0 - 0.25 <= t <= t1 + 0.25] or [l for _, l in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in inside:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes_and_flops(inp):
    """Bytes one call must move at minimum and the FLOPs it must do.

    Bytes: q + every distinct KV row attended (row_bytes each) + the C4 index
    lists + the page-table entries the resolution reads (one per distinct
    page touched per request) + seq_lens (+ cu_seqlens_q) + out + lse.
    FLOPs: 4*H*512 per (token, attended key): QK^T and PV, 2 each per MAC.
    """
    seq = inp.seq_lens.cpu().tolist()
    if inp.cu_seqlens_q is None:
        reqs = list(range(len(seq)))
        poss = [s - 1 for s in seq]
    else:
        cu = inp.cu_seqlens_q.cpu().tolist()
        reqs = [b for b in range(len(seq)) for _ in range(cu[b + 1] - cu[b])]
        poss = [seq[b] - (cu[b + 1] - cu[b]) + i for b in range(len(seq)) for i in range(cu[b + 1] - cu[b])]
    topk = None if inp.topk_idx is None else inp.topk_idx.cpu().tolist()
    T, H = inp.T, inp.H
    w = inp.work
    row_b = 1024 if w.kv_format == "bf16" else 604
    swa_rows, ex_rows, pages = set(), set(), set()
    keys = 0
    for t in range(T):
        b, p = int(reqs[t]), int(poss[t])
        first = max(0, p - w.window + 1)
        for j in range(first, p + 1):
            swa_rows.add((b, j))
            pages.add(("s", b, j // 256))
        n_sw = p + 1 - first
        if w.ratio == 4:
            idx = [int(x) for x in topk[t] if x >= 0]
        elif w.ratio == 128:
            idx = list(range((p + 1) // 128))
        else:
            idx = []
        for i in idx:
            ex_rows.add((b, i))
            pages.add(("e", b, i // 256))
        keys += n_sw + len(idx)
    nbytes = (T * H * 512 * 2 * 2 + T * H * 4 + (len(swa_rows) + len(ex_rows)) * row_b + 4 * len(pages)
              + 4 * w.batch + (0 if inp.topk_idx is None else inp.topk_idx.numel() * 4)
              + (0 if inp.cu_seqlens_q is None else 4 * (w.batch + 1)))
    flops = 4.0 * H * 512 * keys
    return nbytes, flops


def store_algorithmic_bytes(inp):
    """Bytes one cache-write call must move: each new bf16 row read (1024),
    each stored row written (604 for a packed row - the 4 padding bytes are
    not counted - or 1024), its request row and position (8), and one
    page-table entry per distinct (request row, logical page)."""
    n = inp.k.shape[0]
    row_out = 604 if inp.work.kv_format == "fp8" else 1024
    pages = set(zip(inp.req_rows.cpu().tolist(), (inp.positions.cpu() // 256).tolist()))
    return n * (1024 + row_out + 8) + 4 * len(pages)


def is_store_workload(name):
    return name.startswith("kv_store")


def is_topk_workload(name):
    return name.startswith("topk")


def topk_algorithmic_bytes(inp):
    """Bytes one selection call must move: every candidate score read once
    (4 bytes), the lengths, and the k output indices per row."""
    lengths = inp.lengths.cpu().long()
    return int(lengths.sum()) * 4 + 4 * inp.scores.shape[0] + 4 * inp.scores.shape[0] * inp.work.k


# ---------------------------------------------------------------- reference arm (the oracle)
def run_reference_store(args):
    from hybrid_sparse_mqa_gb300 import synth
    from oracle import dsv4_oracle as O
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    inp = synth.make_store_inputs(args.workload, device="cpu")
    kw = inp.oracle_kwargs()
    n = inp.k.shape[0]
    per = min(n, args.ref_rows)
    sl = lambda k: dict(kw, bits=kw["bits"][k:k + per], req_rows=kw["req_rows"][k:k + per],
                        positions=kw["positions"][k:k + per])
    O.kv_store(**sl(0))
    for _ in range(args.warmup):
        O.kv_store(**sl(0))
    t0 = time.perf_counter()
    done = 0
    for k in range(args.steps):
        start = (k * per) % max(1, n - per + 1)
        O.kv_store(**sl(start))
        done += per
    dt = time.perf_counter() - t0
    value = done / dt
    line = {
        "impl": "reference", "metric": STORE_METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "rows_per_step": per,
                   "note": f"oracle sample: {per} of the {n} new rows per step"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} steps x {per} rows of {args.workload}, one process "
                                   f"(the oracle's numpy code runs on one core)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_reference_topk(args):
    from hybrid_sparse_mqa_gb300 import synth
    from oracle import dsv4_oracle as O
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    inp = synth.make_topk_inputs(args.workload, device="cpu")
    kw = inp.oracle_kwargs()
    rows = inp.scores.shape[0]
    per = 1
    O.topk_indices(kw["scores"][:1], kw["lengths"][:1], kw["k"])
    t0 = time.perf_counter()
    for s in range(args.steps):
        r = s % rows
        O.topk_indices(kw["scores"][r:r + 1], kw["lengths"][r:r + 1], kw["k"])
    dt = time.perf_counter() - t0
    value = args.steps * per / dt
    line = {
        "impl": "reference", "metric": TOPK_METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": args.workload, "rows_per_step": per,
                   "note": f"oracle sample: one of the {rows} rows per step"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} rows of {args.workload}, one per step"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_reference(args):
    """The oracle as it stands (numpy float64) on the host's cores: every step
    is a bounded sample of the workload's query tokens spread over one
    spawned process per core (one BLAS thread each)."""
    from hybrid_sparse_mqa_gb300 import synth
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    inp = synth.make_inputs(args.workload, device="cpu")
    T = inp.T
    cores = os.cpu_count() or 1
    per_step_tokens = min(T, max(args.ref_tokens, cores))
    with oracle_pool(inp, cores) as pool:
        def step(k):
            toks = [[(k * per_step_tokens + i) % T] for i in range(per_step_tokens)]
            return sum(pool.map(_oracle_tokens, toks, chunksize=1))
        for w in range(args.warmup):
            step(w)
        t0 = time.perf_counter()
        done = 0
        for k in range(args.steps):
            done += step(k)
        dt = time.perf_counter() - t0
    value = done / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "tokens_per_step": per_step_tokens,
                   "note": f"oracle sample: {per_step_tokens} of the {T} query tokens per step"},
        "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x {per_step_tokens} tokens of {args.workload}, "
                                   f"{cores} spawned processes with one BLAS thread each"},
        "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm: cache write
def run_store(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from hybrid_sparse_mqa_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from hybrid_sparse_mqa_gb300 import attn, synth

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets = rotating_sets(lambda r: synth.make_store_inputs(args.workload, device=dev, seed=2000 * (rank + 1) + r),
                         store_algorithmic_bytes, args.sets, l2)
    pools = [attn.make_pool(s.pool, s.page_table) for s in sets]
    inp0 = sets[0]
    n = inp0.k.shape[0]
    nbytes = store_algorithmic_bytes(inp0)
    R = len(sets)
    stream = torch.cuda.Stream(device=dev)

    def step(k, s=stream):
        i = k % R
        attn.dsv4_kv_store(sets[i].k, sets[i].req_rows, sets[i].positions, pools[i], stream=s)

    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 1)):
            step(k)
    torch.cuda.synchronize()
    if attn.dsv4_attn_get_device_error(stream) != 0:
        raise RuntimeError("device error flags set during warm-up")
    plan, (graph, gcalls) = capture_steps(step, R, args.steps, stream)
    lead = capture_lead(step, R, stream)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if not args.quick:
        clocks.start()
        time.sleep(0.5)
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.5 / max(1e-6, 20e-6 * gcalls)))):
                graph.replay()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream, lead)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        replay(plan)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks.mark()
    clocks.stop()
    ms = slowest_ms(ev0.elapsed_time(ev1), world, dev)
    flags = attn.dsv4_attn_get_device_error(stream)
    sec_per_step = ms / 1e3 / args.steps
    value = job_tokens_per_s(n, world, sec_per_step)

    # ---- end to end: the new rows and their indices from pinned host memory,
    # the store, and the first stored row read back
    pin = lambda x: x.cpu().pin_memory()
    hk = [pin(s.k) for s in sets]
    hreq = [pin(s.req_rows) for s in sets]
    hpos = [pin(s.positions) for s in sets]
    first = []
    for s in sets:
        r, p0 = int(s.req_rows[0]), int(s.positions[0])
        first.append(int(s.page_table[r, p0 // 256]) * 256 + p0 % 256)
    hrow = [torch.empty(s.pool.shape[1:], dtype=s.pool.dtype, pin_memory=True) for s in sets]
    h2d = hk[0].numel() * 2 + hreq[0].numel() * 4 + hpos[0].numel() * 4
    d2h = hrow[0].numel() * hrow[0].element_size()

    def e2e_step(k):
        i = k % R
        s = sets[i]
        s.k.copy_(hk[i], non_blocking=True)
        s.req_rows.copy_(hreq[i], non_blocking=True)
        s.positions.copy_(hpos[i], non_blocking=True)
        attn.dsv4_kv_store(s.k, s.req_rows, s.positions, pools[i], stream=stream)
        hrow[i].copy_(s.pool[first[i]], non_blocking=True)

    e2e_steps = min(args.steps, args.e2e_steps)
    with torch.cuda.stream(stream):
        for k in range(3):
            e2e_step(k)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for k in range(e2e_steps):
            e2e_step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = slowest_ms(e0.elapsed_time(e1), world, dev)
    e2e_value = job_tokens_per_s(n, world, ems / 1e3 / e2e_steps)

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        from oracle import dsv4_oracle as O
        kw = sets[0].oracle_kwargs()
        per = min(n, args.ref_rows)
        sub = dict(kw, bits=kw["bits"][:per], req_rows=kw["req_rows"][:per], positions=kw["positions"][:per])
        O.kv_store(**sub)
        t0 = time.perf_counter()
        done = 0
        while time.perf_counter() - t0 < args.cpu_seconds:
            O.kv_store(**sub)
            done += per
        dt = time.perf_counter() - t0
        cpu_baseline = {"value": done / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
                        "sample": f"{done // per} oracle calls of {per} rows of {args.workload}, {dt:.1f} s, "
                                  f"numpy (pack vectorised, placement one row at a time)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peaks = measured_peaks()
    achieved = nbytes / sec_per_step / 1e9
    w = inp0.work
    line = {
        "metric": STORE_METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "rows": n, "requests": w.requests,
                   "rows_per_request": w.rows_per_request, "kv_format": w.kv_format, "input_sets": R,
                   "l2": f"inputs larger than L2: {R} rotating sets with their own pools "
                         f"({R * nbytes / 1e6:.0f} MB touched per rotation vs L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA-graph replays (one graph for runs of up to 512 steps, else graphs of whole rotations of about 256 calls), step k on input set k mod sets, CUDA events on the launch stream after a 1 ms device spin"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(args.workload),
                     "peak_source": peaks["source"], "algorithmic_bytes_per_launch": nbytes,
                     "us_per_launch": sec_per_step * 1e6},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "cpu_baseline": cpu_baseline,
        "clocks": clocks.summary(),
        "device_error_flags": flags,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- our arm: top-k selection
def run_topk(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from hybrid_sparse_mqa_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from hybrid_sparse_mqa_gb300 import attn, synth

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets = rotating_sets(lambda r: synth.make_topk_inputs(args.workload, device=dev, seed=3000 * (rank + 1) + r),
                         topk_algorithmic_bytes, args.sets, l2)
    inp0 = sets[0]
    rows, k = inp0.scores.shape[0], inp0.work.k
    max_len = int(inp0.lengths.max())
    nbytes = topk_algorithmic_bytes(inp0)
    R = len(sets)
    outs = [torch.empty(rows, k, dtype=torch.int32, device=dev) for _ in sets]
    stream = torch.cuda.Stream(device=dev)

    def step(i, s=stream):
        i %= R
        attn.dsv4_topk(sets[i].scores, sets[i].lengths, k, max_length=max_len, out=outs[i], stream=s)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i)
    torch.cuda.synchronize()
    if attn.dsv4_attn_get_device_error(stream) != 0:
        raise RuntimeError("device error flags set during warm-up")
    plan, (graph, gcalls) = capture_steps(step, R, args.steps, stream)
    lead = capture_lead(step, R, stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if not args.quick:
        clocks.start()
        time.sleep(0.5)
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.5 / max(1e-6, 10e-6 * gcalls)))):
                graph.replay()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream, lead)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        replay(plan)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks.mark()
    clocks.stop()
    ms = slowest_ms(ev0.elapsed_time(ev1), world, dev)
    flags = attn.dsv4_attn_get_device_error(stream)
    sec_per_step = ms / 1e3 / args.steps
    value = job_tokens_per_s(rows, world, sec_per_step)

    # ---- end to end: scores and lengths from pinned host memory, the call,
    # the index lists back to pinned host memory
    hs = [s.scores.cpu().pin_memory() for s in sets]
    hl = [s.lengths.cpu().pin_memory() for s in sets]
    ho = [torch.empty(rows, k, dtype=torch.int32, pin_memory=True) for _ in sets]
    h2d = hs[0].numel() * 4 + hl[0].numel() * 4
    d2h = ho[0].numel() * 4

    def e2e_step(i):
        i %= R
        sets[i].scores.copy_(hs[i], non_blocking=True)
        sets[i].lengths.copy_(hl[i], non_blocking=True)
        step(i)
        ho[i].copy_(outs[i], non_blocking=True)

    e2e_steps = min(args.steps, args.e2e_steps)
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = slowest_ms(e0.elapsed_time(e1), world, dev)
    e2e_value = job_tokens_per_s(rows, world, ems / 1e3 / e2e_steps)

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        from oracle import dsv4_oracle as O
        kw = sets[0].oracle_kwargs()
        O.topk_indices(kw["scores"][:1], kw["lengths"][:1], k)
        t0 = time.perf_counter()
        done = 0
        while time.perf_counter() - t0 < args.cpu_seconds:
            r = done % rows
            O.topk_indices(kw["scores"][r:r + 1], kw["lengths"][r:r + 1], k)
            done += 1
        dt = time.perf_counter() - t0
        cpu_baseline = {"value": done / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
                        "sample": f"{done} rows of {args.workload}, one oracle call each, {dt:.1f} s "
                                  f"(a Python sort per row: one core)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peaks = measured_peaks()
    achieved = nbytes / sec_per_step / 1e9
    line = {
        "metric": TOPK_METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": args.workload, "rows": rows, "candidates_per_row": max_len, "k": k,
                   "input_sets": R,
                   "l2": f"inputs larger than L2: {R} rotating sets ({R * nbytes / 1e6:.0f} MB touched per "
                         f"rotation vs L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA-graph replays (one graph for runs of up to 512 steps, else graphs of whole rotations of about 256 calls), step k on input set k mod sets, CUDA events on the launch stream after a 1 ms device spin"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(args.workload),
                     "peak_source": peaks["source"], "algorithmic_bytes_per_launch": nbytes,
                     "us_per_launch": sec_per_step * 1e6},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "cpu_baseline": cpu_baseline,
        "clocks": clocks.summary(),
        "device_error_flags": flags,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- our arm
SECOND_WORKLOAD = "c128_decode"     # the other decode configuration with a roofline target


def measure_workload(args, workload, dev, world, steps):
    """Times `steps` calls of `workload` exactly as the headline line does
    (rotating input sets with their own pools, CUDA-graph replays on a busy
    stream, CUDA events on the launch stream, slowest rank) and returns its
    entry: throughput and the roofline of one call."""
    import torch
    from hybrid_sparse_mqa_gb300 import attn, synth
    rank, _, _ = dist_env()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets = rotating_sets(lambda r: synth.make_inputs(workload, device=dev, seed=2000 * (rank + 1) + r),
                         lambda x: algorithmic_bytes_and_flops(x)[0], args.sets, l2)
    inp0 = sets[0]
    T, H = inp0.T, inp0.H
    w = inp0.work
    nbytes, flops = algorithmic_bytes_and_flops(inp0)
    outs = [torch.empty_like(x.q) for x in sets]
    lses = [torch.empty(T, H, dtype=torch.float32, device=dev) for _ in sets]
    topk = w.topk if w.ratio == 4 else 0
    sc, sg = attn.dsv4_attn_plan(T, H, w.ratio, w.window, topk, inp0.max_seq_len, 0)
    wsz = attn.dsv4_attn_workspace_size(T, H, w.ratio, w.window, topk, inp0.max_seq_len, 0)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(k, st):
        i = k % len(sets)
        attn.run_inputs(sets[i], out=outs[i], lse=lses[i], workspace=ws, stream=st)

    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 1)):
            step(k, stream)
    torch.cuda.synchronize()
    R = len(sets)
    plan, (graph, gcalls) = capture_steps(step, R, steps, stream)
    lead = capture_lead(step, R, stream)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream, lead)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        replay(plan)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = slowest_ms(ev0.elapsed_time(ev1), world, dev)
    flags = attn.dsv4_attn_get_device_error(stream)
    sec = ms / 1e3 / steps
    peaks = measured_peaks()
    achieved = nbytes / sec / 1e9
    tflops = flops / sec / 1e12
    tensor_bound = flops / (peaks["bf16_tflops"] * 1e12) > nbytes / (peaks["hbm_gbs"] * 1e9)
    return {
        "value": job_tokens_per_s(T, world, sec), "unit": "query-tokens/s", "ms_per_step": sec * 1e3,
        "steps": steps, "device_error_flags": flags,
        "config": {"workload": workload, "batch": w.batch, "heads": H, "context": int(inp0.max_seq_len),
                   "split_plan": {"cluster_splits": sc, "grid_splits": sg}, "input_sets": R},
        "gpu_launches": steps * (2 if sg > 1 else 1),
        "roofline": {"bound": "tensor" if tensor_bound else "hbm",
                     "achieved": tflops if tensor_bound else achieved,
                     "peak": peaks["bf16_tflops"] if tensor_bound else peaks["hbm_gbs"],
                     "unit": "TFLOP/s" if tensor_bound else "GB/s",
                     "frac": tflops / peaks["bf16_tflops"] if tensor_bound else achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(workload), "peak_source": peaks["source"],
                     "algorithmic_bytes_per_launch": nbytes, "flops_per_launch": flops,
                     "hbm_gbs": achieved, "hbm_frac": achieved / peaks["hbm_gbs"],
                     "tensor_tflops": tflops, "tensor_frac": tflops / peaks["bf16_tflops"],
                     "us_per_launch": sec * 1e6},
    }


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from hybrid_sparse_mqa_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    from hybrid_sparse_mqa_gb300 import attn, synth

    # ---- rotating input sets, each with its own pools: the data one step
    # reads was last touched R steps earlier, so it is not in L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets = rotating_sets(lambda r: synth.make_inputs(args.workload, device=dev, seed=1000 * (rank + 1) + r),
                         lambda x: algorithmic_bytes_and_flops(x)[0], args.sets, l2)
    inp0 = sets[0]
    T, H = inp0.T, inp0.H
    nbytes, flops = algorithmic_bytes_and_flops(inp0)
    outs = [torch.empty_like(s.q) for s in sets]
    lses = [torch.empty(T, H, dtype=torch.float32, device=dev) for _ in sets]
    w = inp0.work
    sc, sg = attn.dsv4_attn_plan(T, H, w.ratio, w.window, w.topk if w.ratio == 4 else 0, inp0.max_seq_len,
                                 args.num_splits)
    wsz = attn.dsv4_attn_workspace_size(T, H, w.ratio, w.window, w.topk if w.ratio == 4 else 0,
                                        inp0.max_seq_len, args.num_splits)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device=dev)
    launches_per_step = 1 + (1 if sg > 1 else 0)
    stream = torch.cuda.Stream(device=dev)

    def step(k, s=stream):
        i = k % len(sets)
        attn.run_inputs(sets[i], out=outs[i], lse=lses[i], workspace=ws, stream=s, num_splits=args.num_splits)

    # ---- warm-up (also warms the library's per-device cache before capture)
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 1)):
            step(k)
    torch.cuda.synchronize()
    if attn.dsv4_attn_get_device_error(stream) != 0:
        raise RuntimeError("device error flags set during warm-up")

    # ---- one CUDA graph holds one call per input set; replays cover K steps
    R = len(sets)
    plan, (graph, gcalls) = capture_steps(step, R, args.steps, stream)
    lead = capture_lead(step, R, stream)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if not args.quick:
        clocks.start()
        time.sleep(0.5)
        # spin the GPU for a moment so the clock samples see it under load
        with torch.cuda.stream(stream):
            for _ in range(max(1, int(0.5 / max(1e-6, 6e-6 * gcalls)))):
                graph.replay()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream, lead)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        replay(plan)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks.mark()
    clocks.stop()
    ms = slowest_ms(ev0.elapsed_time(ev1), world, dev)
    flags = attn.dsv4_attn_get_device_error(stream)
    sec_per_step = ms / 1e3 / args.steps
    value = job_tokens_per_s(T, world, sec_per_step)

    # ---- per launch: the binding called once per step, no CUDA graph (the
    # host's launch overhead counts wherever it exceeds the kernel's time)
    n_eager = max(1, min(args.steps, 200))
    torch.cuda.synchronize()
    ea0, ea1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea0.record(stream)
    for k in range(n_eager):
        step(k, stream)
    ea1.record(stream)
    torch.cuda.synchronize()
    eager_us = slowest_ms(ea0.elapsed_time(ea1), world, dev) * 1e3 / n_eager
    flags |= attn.dsv4_attn_get_device_error(stream)

    # ---- end to end through the public API with host buffers
    pin = lambda x: x.cpu().pin_memory()
    hq = [pin(s.q) for s in sets]
    hidx = [pin(s.topk_idx) if s.topk_idx is not None else None for s in sets]
    hseq = [pin(s.seq_lens) for s in sets]
    hout = [torch.empty(T, H, 512, dtype=torch.bfloat16).pin_memory() for _ in sets]
    hlse = [torch.empty(T, H, dtype=torch.float32).pin_memory() for _ in sets]
    h2d = hq[0].numel() * 2 + hseq[0].numel() * 4 + (0 if hidx[0] is None else hidx[0].numel() * 4)
    d2h = hout[0].numel() * 2 + hlse[0].numel() * 4

    def e2e_step(k):
        i = k % R
        s = sets[i]
        s.q.copy_(hq[i], non_blocking=True)
        s.seq_lens.copy_(hseq[i], non_blocking=True)
        if hidx[i] is not None:
            s.topk_idx.copy_(hidx[i], non_blocking=True)
        attn.run_inputs(s, out=outs[i], lse=lses[i], workspace=ws, stream=stream, num_splits=args.num_splits)
        hout[i].copy_(outs[i], non_blocking=True)
        hlse[i].copy_(lses[i], non_blocking=True)

    e2e_steps = min(args.steps, args.e2e_steps)
    with torch.cuda.stream(stream):
        for k in range(3):
            e2e_step(k)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for k in range(e2e_steps):
            e2e_step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = slowest_ms(e0.elapsed_time(e1), world, dev)
    e2e_value = job_tokens_per_s(T, world, ems / 1e3 / e2e_steps)

    # ---- the other decode configuration with a roofline target, timed the same way
    second = None
    if args.workload == DEFAULT_WORKLOAD and args.num_splits == 0 and not args.no_second:
        second = measure_workload(args, SECOND_WORKLOAD, dev, world, args.steps)

    # ---- oracle on the host, bounded sample of the same workload (rank 0, N=1)
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        inp_cpu = synth.make_inputs(args.workload, device="cpu", seed=1000 * (rank + 1))
        cores = os.cpu_count() or 1
        v_all, n_all = oracle_throughput(inp_cpu, cores, args.cpu_seconds / 6)
        v_one, n_one = oracle_throughput(inp_cpu, 1, args.cpu_seconds / 6)
        cpu_baseline = {"value": v_all, "unit": "query-tokens/s", "cores": cores, "kind": "oracle",
                        "one_core": v_one,
                        "sample": f"{args.workload} query tokens, numpy float64, tasks of 4 tokens: {cores} spawned "
                                  f"processes with one BLAS thread each ({n_all} tokens per run) and 1 process "
                                  f"({n_one} tokens per run), best of 3 runs each"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peaks = measured_peaks()
    per_launch_s = sec_per_step / launches_per_step if launches_per_step == 1 else sec_per_step
    achieved = nbytes / per_launch_s / 1e9
    tflops = flops / per_launch_s / 1e12
    # the roofline that binds: bytes at the HBM peak or FLOPs at the bf16
    # tensor peak (the burst figure: the kernel is timed on its own)
    tensor_bound = flops / (peaks["bf16_tflops"] * 1e12) > nbytes / (peaks["hbm_gbs"] * 1e9)
    roofline = {"bound": "tensor" if tensor_bound else "hbm",
                "achieved": tflops if tensor_bound else achieved,
                "peak": peaks["bf16_tflops"] if tensor_bound else peaks["hbm_gbs"],
                "unit": "TFLOP/s" if tensor_bound else "GB/s",
                "frac": tflops / peaks["bf16_tflops"] if tensor_bound else achieved / peaks["hbm_gbs"],
                "traffic": ncu_traffic(args.workload), "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": nbytes, "flops_per_launch": flops,
                "hbm_gbs": achieved, "hbm_frac": achieved / peaks["hbm_gbs"],
                "hbm_frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "tensor_tflops": tflops, "tensor_frac": tflops / peaks["bf16_tflops"],
                "us_per_launch": per_launch_s * 1e6}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "query-tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": w.batch, "heads": H, "head_dim": 512,
                   "context": int(inp0.max_seq_len), "topk": w.topk if w.ratio == 4 else 0,
                   "window": w.window, "input_sets": R,
                   "l2": f"inputs larger than L2: {R} rotating sets with their own pools "
                         f"({R * nbytes / 1e6:.0f} MB touched per rotation vs L2 {l2 / 1e6:.0f} MB)",
                   "split_plan": {"cluster_splits": sc, "grid_splits": sg},
                   "timing": "CUDA-graph replays (one graph for runs of up to 512 steps, else graphs of whole rotations of about 256 calls), step k on input set k mod sets, CUDA events on the launch stream after a 1 ms device spin"},
        "gpu_launches": args.steps * launches_per_step,
        "roofline": roofline,
        "per_launch": {"us_per_call": eager_us, "calls": n_eager,
                       "timing": "eager calls of the Python binding one after another on the launch stream, "
                                 "no CUDA graph; CUDA events"},
        "e2e": {"value": e2e_value, "unit": "query-tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "cpu_baseline": cpu_baseline,
        "clocks": clocks.summary(),
        "device_error_flags": flags,
    }
    if second is not None:
        line[SECOND_WORKLOAD] = second
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sets", type=int, default=0,
                    help="input sets in the timed rotation (0: at least 12 and four times the L2 per rotation)")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="key-list pieces per token (0 = the library's plan)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--ref-rows", type=int, default=4096,
                    help="rows per oracle call for the cache-write workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-second", action="store_true",
                    help=f"skip the {SECOND_WORKLOAD} entry of the default line")
    ap.add_argument("--quick", action="store_true",
                    help="no clock sampling, no CPU baseline (for profiler runs)")
    args = ap.parse_args()
    if is_store_workload(args.workload):
        return run_reference_store(args) if args.impl == "reference" else run_store(args)
    if is_topk_workload(args.workload):
        return run_reference_topk(args) if args.impl == "reference" else run_topk(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
