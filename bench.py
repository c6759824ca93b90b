#!/usr/bin/env python3
"""Benchmark: paged decode attention on one GB300.

One step is one paged_decode_attention call on the long-context GQA decode of
the kernel-latency table of "[Performance] Support MQA/GQA in decode phase by
using FlashAttention" (context_len 4096, batch 256 row): 256 sequences, 64
query heads on 8 KV heads, head_size 128, block_size 16, bf16, every
sequence 4096 tokens through a seeded random block table over a 65536-block
pool (4.3 GB of K and V).  The call covers address translation, query
staging, both products, the online softmax, split-context partials and their
log-sum-exp merge: the library plans the split, and at this size it takes
the stream form (every SM an equal share of all tiles, cut pairs merged by a
second launch).

Prints ONE JSON line (rank 0).  `value` is algorithmic HBM bytes per step
(K and V of every cached token, q read, out written, block-table entries and
lengths) divided by device time per step, GB/s (1e9).  The KV pool is 33x
the L2, so every step streams its inputs from HBM.  Beside it: `e2e` (the
same call with q, tables and lengths copied in from pinned host memory and
out copied back, every step, the steps pipelined as a serving loop runs
them: one step's copies overlap the neighbouring steps' calls), `roofline`
against the measured copy
bandwidth, `cpu_baseline` (the float64 oracle on a sample of the same
workload, one core and all cores), and side lines for the other decode
workloads, gather_cached_kv and prefill.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkd|reference]
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# The oracle runs one BLAS thread per process (the all-core leg uses one
# process per core); set before NumPy loads its BLAS.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

METRIC = ("paged decode attn µs/call and achieved HBM GB/s (% of GB300 roofline) "
          "vs oracle")
HEADLINE = "gqa_ctx4096_b256"
HEADLINE_DESC = "S=256 H=64 Hk=8 D=128 B=16 ctx=4096 NB=65536 bf16"
# Side lines, decode alone: the other decode workloads at batch >= 64 and
# context >= 1024, and the LLaMA-13B MHA decode.
SIDE_DECODE = ["gqa_ctx1024_b64", "gqa_ctx1024_b256", "gqa_ctx4096_b64", "mqa_ragged_b64",
               "llama13b_mha_b8_ctx256"]
SIDE_GATHER = "gather_t2048"
PATH_NAMES = {0: "simt", 1: "tc", 2: "tc_cluster", 3: "tc_stream"}   # decode_plan's kernel family
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# ncu DRAM traffic per launch, stored with the hash of the sources it was
# measured on; reported only while those sources are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
DECODE_SOURCES = ("paged_kv_decode_22_gb300/csrc/decode_tc.cu",
                  "paged_kv_decode_22_gb300/csrc/lse_reduce.cu",
                  "paged_kv_decode_22_gb300/csrc/schedule.cuh",
                  "paged_kv_decode_22_gb300/csrc/sm100.cuh",
                  "paged_kv_decode_22_gb300/csrc/common.cuh",
                  "paged_kv_decode_22_gb300/csrc/internal.h",
                  "paged_kv_decode_22_gb300/csrc/api.cu")


def max_over_ranks(ms, dist, device):
    """Step time of the slowest rank (every rank gets it); `dist` is
    torch.distributed or None for a single process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(step_bytes, world, ms):
    """Whole-job throughput: every rank processed step_bytes per step, timed
    by the slowest rank (weak scaling: the per-GPU work is fixed)."""
    return step_bytes * world / ms / 1e6


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


# ---------------------------------------------------------------- byte counts

def decode_bytes(c) -> int:
    """Algorithmic HBM bytes of one decode call: K+V rows read, q read, out
    written, block-table entries and context lengths read."""
    e = 2
    lens = [int(x) for x in c.context_lens]
    kv = sum(lens) * c.num_kv_heads * c.head_size * 2 * e
    qo = 2 * c.num_seqs * c.num_heads * c.head_size * e
    tables = 4 * sum(-(-L // c.block_size) for L in lens) + 4 * c.num_seqs
    return kv + qo + tables


def gather_bytes(g) -> int:
    """K and V rows read and written once each, plus the slot mapping."""
    return 2 * 2 * g.num_tokens * g.num_heads * g.head_size * 2 + 8 * g.num_tokens


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="pkd_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        busy = [v for v in sm if mx and v >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def src_hash(rel_paths):
    h = hashlib.sha256()
    for r in rel_paths:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(key, rel_paths):
    """DRAM bytes per launch recorded for `key` in the traffic file, or None
    when there is none or the sources changed since it was measured."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources_sha256_16") != src_hash(rel_paths):
        return None
    return rec.get("dram_bytes_per_launch")


def peaks():
    """(HBM GB/s, its source, bf16 TF/s burst) from MEASURED_PEAKS.json."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, src, tf = FALLBACK_HBM_GBS, "fallback", FALLBACK_BF16_TFLOPS
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        if pk.get("hbm_gbs"):
            hbm, src = float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
        if pk.get("bf16_tflops"):
            tf = float(pk["bf16_tflops"])
    return hbm, src, tf


def timed_loop(call, steps, mark):
    """The timed region: mark(0), exactly `steps` calls, mark(1)."""
    mark(0)
    for _ in range(steps):
        call()
    mark(1)


def preroll_calls(call_us, window_s=0.6, cap=20000):
    """Untimed calls that keep the GPU busy for about `window_s` before the
    timed region, so that the clock samples see it under load."""
    if not call_us or call_us <= 0:
        return 0
    return int(min(cap, math.ceil(window_s * 1e6 / call_us)))


# ---------------------------------------------------------------- oracle (CPU baseline, reference arm)

_ORACLE = {}


def _oracle_sample_case(name, nseq):
    """A sample of workload `name`: its first `nseq` sequences (lengths, head
    shape, block size, dtype), on a pool of just the blocks they need."""
    from paged_kv_decode_22_gb300.workloads import decode_configs, make_decode_case
    cfg = dict(decode_configs()[name])
    lens = [int(x) for x in cfg["context_lens"]][:nseq]
    need = sum(-(-L // cfg["block_size"]) for L in lens)
    cfg.update(num_seqs=len(lens), context_lens=lens, num_blocks=need, poison=False)
    return make_decode_case(name=f"{name}[:{len(lens)}]", **cfg)


def _oracle_init(name, nseq):
    _ORACLE["case"] = _oracle_sample_case(name, nseq)


def _oracle_pass(_=None):
    """One oracle pass over the worker's sample: (seconds, bytes)."""
    from oracle.paged_attention import paged_decode_attention as ref_attn
    c = _ORACLE["case"]
    t0 = time.perf_counter()
    ref_attn(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens, c.scale, c.dtype)
    return time.perf_counter() - t0, decode_bytes(c)


def _oracle_budget(budget_s):
    """Oracle passes over the worker's sample until budget_s has elapsed:
    (bytes processed, seconds, passes)."""
    _oracle_pass()                       # first touch of the sample's pages
    nbytes, n, t0 = 0, 0, time.perf_counter()
    while True:
        _, b = _oracle_pass()
        nbytes += b
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return nbytes, el, n


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pool(procs, name, nseq):
    """`procs` spawned worker processes (one BLAS thread each), each holding
    its own copy of the sample.  Spawned, so safe after CUDA is initialised."""
    import multiprocessing as mp
    return mp.get_context("spawn").Pool(procs, initializer=_oracle_init, initargs=(name, nseq))


def cpu_baseline(name, budget_s=8.0, nseq=2):
    """The oracle as it stands on this host's cores, on a bounded sample of
    workload `name`: one process, then one process per core, each timing
    passes over its own `nseq`-sequence sample for about budget_s."""
    cores = host_cores()
    _oracle_init(name, nseq)
    b1, t1, n1 = _oracle_budget(budget_s)
    one = round(b1 / t1 / 1e9, 4)
    with oracle_pool(cores, name, nseq) as pool:
        res = pool.map(_oracle_budget, [budget_s] * cores)
    ball = sum(r[0] for r in res)
    tall = max(r[1] for r in res)
    allv = round(ball / tall / 1e9, 4)
    what = (f"{name}: sequences 0..{nseq - 1} of the workload (same head shape, block size, "
            f"context and dtype) per process, float64 oracle passes for ~{budget_s:.0f} s")
    return {"value": allv, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{what}; {sum(r[2] for r in res)} passes over {cores} processes",
            "single_core": {"value": one, "unit": "GB/s", "cores": 1, "passes": n1}}


def run_reference(args, world, rank):
    """The oracle as it stands, timed on the host cores, as the reference arm:
    each step is one oracle pass per core over a sample of the headline
    workload, in parallel (one spawned process per core)."""
    if rank != 0:
        return 0
    cores = host_cores()
    # Size each process's sample so that warm-up + timed steps take ~60 s.
    _oracle_init(HEADLINE, 1)
    _oracle_pass()
    t_seq = min(_oracle_pass()[0] for _ in range(2))
    nseq = int(max(1, min(16, 60.0 / max(1, args.steps + args.warmup) / t_seq)))
    with oracle_pool(cores, HEADLINE, nseq) as pool:
        pool.map(_oracle_pass, range(cores))          # every worker built and warm
        for _ in range(args.warmup):
            pool.map(_oracle_pass, range(cores))
        nbytes, t0 = 0, time.perf_counter()
        for _ in range(args.steps):
            nbytes += sum(r[1] for r in pool.map(_oracle_pass, range(cores)))
        dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / args.steps / dt / 1e9
    what = (f"{HEADLINE}: per step, one float64 oracle pass over sequences 0..{nseq - 1} of the "
            f"workload in each of {cores} processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs, random non-overlapping block tables)",
        "config": {"workload": HEADLINE, "shape": HEADLINE_DESC, "sample": what},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": what},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def graph_time(fns, calls=32, reps=5):
    """Mean device time per call (us) of the calls fns[i % len(fns)], replayed
    as one CUDA graph of `calls` calls."""
    import torch
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for i in range(calls):
            fns[i % len(fns)]()
    gr.replay()
    gr.replay()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        gr.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * calls)


def time_decode_workload(name, dev, ops, partition_size=0):
    """(us per call, algorithmic bytes, plan) of one decode workload, inputs
    rotated over enough copies to exceed 3x L2; partition_size as in
    paged_decode_attention (0: the library's plan)."""
    import torch
    d0 = device_decode_inputs(name, dev)
    S, H, D = d0["q"].shape
    Hk, B = d0["kc"].shape[2], d0["kc"].shape[1]
    ncopy = max(1, min(8, math.ceil(3 * L2_BYTES / d0["bytes"])))
    sets = [d0] + [dict(d0, q=d0["q"].clone(), kc=d0["kc"].clone(), vc=d0["vc"].clone(),
                        out=torch.empty_like(d0["out"])) for _ in range(ncopy - 1)]
    plan = ops.decode_plan(S, H, Hk, D, B, d0["max_ctx"], partition_size)
    work = torch.empty(max(plan[3], 256), dtype=torch.uint8, device=dev)
    fns = [lambda d=d: ops.paged_decode_attention(d["out"], d["q"], d["kc"], d["vc"], d["bt"],
                                                  d["cl"], d["max_ctx"], d["scale"],
                                                  partition_size=partition_size,
                                                  workspace=work) for d in sets]
    us = graph_time(fns)
    nbytes = d0["bytes"]
    del d0, sets, work, fns
    torch.cuda.empty_cache()
    return us, nbytes, plan, ncopy


def device_decode_inputs(name, dev, tight=False):
    """Device inputs of a decode workload from a seeded torch generator (for
    timing and profiling: the kernels' speed does not depend on the values).
    tight: a pool of just the blocks the sequences use (small ncu captures)."""
    import torch

    from paged_kv_decode_22_gb300.workloads import decode_configs
    cfg = decode_configs()[name]
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg["seed"])
    S, H, Hk, D, B = (cfg["num_seqs"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_size"],
                      cfg["block_size"])
    lens = torch.tensor(cfg["context_lens"], dtype=torch.int32)
    need = (lens + B - 1) // B
    nb = int(need.sum()) if tight else max(cfg["num_blocks"], int(need.sum()))
    dt = torch.float16 if cfg["dtype"] == "fp16" else torch.bfloat16
    kc = torch.randn((nb, B, Hk, D), generator=gen, device=dev, dtype=dt)
    vc = torch.randn((nb, B, Hk, D), generator=gen, device=dev, dtype=dt)
    q = torch.randn((S, H, D), generator=gen, device=dev, dtype=dt)
    perm = torch.randperm(nb, generator=gen, device=dev).to(torch.int32)
    mb = int(need.max())
    bt = torch.zeros((S, mb), dtype=torch.int32, device=dev)
    pos = 0
    for s in range(S):
        n = int(need[s])
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    nbytes = (int(lens.sum()) * Hk * D * 2 * 2 + 2 * S * H * D * 2 + 4 * int(need.sum()) + 4 * S)
    return dict(q=q, kc=kc, vc=vc, bt=bt, cl=lens.to(dev), max_ctx=int(lens.max()),
                scale=1.0 / math.sqrt(D), out=torch.empty_like(q), bytes=nbytes)


def prefill_work(lens, qlens, H, Hk, D):
    """(causal FLOPs, algorithmic bytes) of one prefill call: each query at
    position p costs 4*D FLOPs per visible token and head (q.K and p.V);
    bytes are every sequence's K/V read once plus q read and out written."""
    flops = 0
    for L, n in zip(lens, qlens):
        vis = n * (L - n) + n * (n + 1) // 2          # sum over queries of (p + 1)
        flops += 4 * D * H * vis
    kv = sum(lens) * Hk * D * 2 * 2
    qo = 2 * sum(qlens) * H * D * 2
    return flops, kv + qo


def device_prefill_inputs(name, dev):
    """Device inputs of a prefill workload from a seeded torch generator."""
    import torch

    from paged_kv_decode_22_gb300.workloads import prefill_configs
    cfg = prefill_configs()[name]
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg["seed"])
    S, H, Hk, D, B = (cfg["num_seqs"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_size"],
                      cfg["block_size"])
    lens = torch.tensor(cfg["context_lens"], dtype=torch.int32)
    qlens = torch.tensor(cfg["query_lens"], dtype=torch.int32)
    need = (lens + B - 1) // B
    nb = max(cfg["num_blocks"], int(need.sum()))
    dt = torch.float16 if cfg["dtype"] == "fp16" else torch.bfloat16
    T = int(qlens.sum())
    kc = torch.randn((nb, B, Hk, D), generator=gen, device=dev, dtype=dt)
    vc = torch.randn((nb, B, Hk, D), generator=gen, device=dev, dtype=dt)
    q = torch.randn((T, H, D), generator=gen, device=dev, dtype=dt)
    perm = torch.randperm(nb, generator=gen, device=dev).to(torch.int32)
    bt = torch.zeros((S, int(need.max())), dtype=torch.int32, device=dev)
    pos = 0
    for si in range(S):
        n = int(need[si])
        bt[si, :n] = perm[pos:pos + n]
        pos += n
    qs = torch.zeros(S + 1, dtype=torch.int32)
    qs[1:] = torch.cumsum(qlens, 0)
    flops, nbytes = prefill_work(lens.tolist(), qlens.tolist(), H, Hk, D)
    return dict(q=q, kc=kc, vc=vc, bt=bt, cl=lens.to(dev), qs=qs.to(dev), max_q=int(qlens.max()),
                max_ctx=int(lens.max()), scale=1.0 / math.sqrt(D), out=torch.empty_like(q),
                flops=flops, bytes=nbytes)


def time_prefill_workload(name, dev, ops):
    """(us per call, FLOPs, bytes, copies) of one prefill workload, inputs
    rotated over enough copies to exceed 3x L2."""
    import torch
    d0 = device_prefill_inputs(name, dev)
    ncopy = max(1, min(8, math.ceil(3 * L2_BYTES / d0["bytes"])))
    sets = [d0] + [dict(d0, q=d0["q"].clone(), kc=d0["kc"].clone(), vc=d0["vc"].clone(),
                        out=torch.empty_like(d0["out"])) for _ in range(ncopy - 1)]
    fns = [lambda d=d: ops.paged_prefill_attention(d["out"], d["q"], d["kc"], d["vc"], d["bt"],
                                                   d["cl"], d["qs"], d["max_q"], d["max_ctx"],
                                                   d["scale"]) for d in sets]
    us = graph_time(fns)
    out = (us, d0["flops"], d0["bytes"], ncopy)
    del d0, sets, fns
    torch.cuda.empty_cache()
    return out


def run_profile(args, local):
    """Run one kernel family on one workload (no timing): the command ncu wraps."""
    import torch

    from paged_kv_decode_22_gb300 import ops
    from paged_kv_decode_22_gb300.workloads import gather_sweep, make_gather_case
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kind, name = args.profile.split(":", 1)
    if kind == "decode":
        d = device_decode_inputs(name, dev, tight=args.tight_pool)
        S, H, D = d["q"].shape
        _, npart, _, ws = ops.decode_plan(S, H, d["kc"].shape[2], D, d["kc"].shape[1],
                                          d["max_ctx"], args.partition_size)
        work = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)

        def call():
            ops.paged_decode_attention(d["out"], d["q"], d["kc"], d["vc"], d["bt"], d["cl"],
                                       d["max_ctx"], d["scale"], workspace=work,
                                       partition_size=args.partition_size)
    elif kind == "prefill":
        d = device_prefill_inputs(name, dev)

        def call():
            ops.paged_prefill_attention(d["out"], d["q"], d["kc"], d["vc"], d["bt"], d["cl"],
                                        d["qs"], d["max_q"], d["max_ctx"], d["scale"])
    elif kind == "gather":
        g = make_gather_case(name=name, **gather_sweep()[name])
        import numpy as np
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.float16).to(dev)
        kc, vc = up(g.key_cache), up(g.value_cache)
        slots = torch.from_numpy(g.slot_mapping).to(dev)
        ko = torch.empty((g.num_tokens, g.num_heads, g.head_size), dtype=torch.float16,
                         device=dev)
        vo = torch.empty_like(ko)

        def call():
            ops.gather_cached_kv(ko, vo, kc, vc, slots)
    else:
        raise SystemExit(f"unknown profile kind {kind}")
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    print(f"profile {args.profile}: {args.warmup + args.steps} calls ok")
    return 0


def run_sweep(args, local):
    """Per-workload device time per call: CUDA-graph replays of 32 calls that
    rotate over enough input copies to exceed 3x L2 (the same method as the
    timed region of the default run)."""
    import torch

    from paged_kv_decode_22_gb300 import ops
    from paged_kv_decode_22_gb300.workloads import (decode_configs, gather_sweep,
                                                    make_gather_case, prefill_configs)
    import numpy as np
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peak = FALLBACK_HBM_GBS
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        with open(pk_path) as f:
            peak = float(json.load(f).get("hbm_gbs") or peak)
    for name in decode_configs():
        try:
            us, nbytes, (ps, npart, path, _), ncopy = time_decode_workload(
                name, dev, ops, args.partition_size)
        except ops.PkdError as e:        # a forced partition size this workload cannot take
            print(json.dumps({"workload": name, "kind": "decode", "skipped": str(e)}), flush=True)
            continue
        print(json.dumps({"workload": name, "kind": "decode", "us_per_call": round(us, 2),
                          "GBps": round(nbytes / us / 1e3, 1),
                          "frac": round(nbytes / us / 1e3 / peak, 3),
                          "path": PATH_NAMES[path], "partitions": npart,
                          "partition_size": ps, "bytes": nbytes, "copies": ncopy}), flush=True)
    tpeak = None
    if os.path.exists(pk_path):
        with open(pk_path) as f:
            tpeak = json.load(f).get("bf16_tflops")
    tpeak = float(tpeak or FALLBACK_BF16_TFLOPS)
    for name in prefill_configs():
        us, flops, nbytes, ncopy = time_prefill_workload(name, dev, ops)
        tf = flops / us / 1e6
        print(json.dumps({"workload": name, "kind": "prefill", "us_per_call": round(us, 2),
                          "TFLOPs": round(tf, 1), "frac_tensor": round(tf / tpeak, 3),
                          "GBps": round(nbytes / us / 1e3, 1),
                          "frac_hbm": round(nbytes / us / 1e3 / peak, 3), "flops": flops,
                          "bytes": nbytes, "copies": ncopy}), flush=True)
    for name, cfg in gather_sweep().items():
        g = make_gather_case(name=name, **cfg)
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.float16).to(dev)
        nb = gather_bytes(g)
        ncopy = max(1, min(8, math.ceil(3 * L2_BYTES / nb)))
        sets = []
        for _ in range(ncopy):
            ko = torch.empty((g.num_tokens, g.num_heads, g.head_size), dtype=torch.float16,
                             device=dev)
            sets.append((ko, torch.empty_like(ko), up(g.key_cache), up(g.value_cache),
                         torch.from_numpy(g.slot_mapping).to(dev)))
        fns = [lambda t=t: ops.gather_cached_kv(*t) for t in sets]
        us = graph_time(fns)
        print(json.dumps({"workload": name, "kind": "gather", "us_per_call": round(us, 2),
                          "GBps": round(nb / us / 1e3, 1), "frac": round(nb / us / 1e3 / peak, 3),
                          "pages_GiBps_one_way": round(nb / 2 / us / 1e3 * 1e9 / 2 ** 30, 1),
                          "bytes": nb, "copies": ncopy}), flush=True)
        del sets, fns
        torch.cuda.empty_cache()
    return 0



def decode_launches(npart, path):
    """Kernel launches of one decode call under its plan: the stream form and
    a split workspace plan add a merge launch; the cluster form merges in
    place."""
    if path == 3 or (path in (0, 1) and npart > 1):
        return 2
    return 1


def side_lines(dev, ops, peak):
    """Graph-timed side lines: decode workloads, gather, prefill."""
    import numpy as np
    import torch

    from paged_kv_decode_22_gb300.workloads import gather_sweep, make_gather_case, prefill_configs
    out = {"decode": {}, "gather": {}, "prefill": {}}
    for name in SIDE_DECODE:
        us, nbytes, (ps, npx, pathx, _), ncopy = time_decode_workload(name, dev, ops)
        out["decode"][name] = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                               "frac": round(nbytes / us / 1e3 / peak, 3),
                               "path": PATH_NAMES[pathx], "partitions": npx, "copies": ncopy}
    g = make_gather_case(name=SIDE_GATHER, **gather_sweep()[SIDE_GATHER])
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.float16).to(dev)
    nb = gather_bytes(g)
    ncopy = max(1, min(8, math.ceil(3 * L2_BYTES / nb)))
    sets = []
    for _ in range(ncopy):
        ko = torch.empty((g.num_tokens, g.num_heads, g.head_size), dtype=torch.float16, device=dev)
        sets.append((ko, torch.empty_like(ko), up(g.key_cache), up(g.value_cache),
                     torch.from_numpy(g.slot_mapping).to(dev)))
    us = graph_time([lambda t=t: ops.gather_cached_kv(*t) for t in sets])
    out["gather"][SIDE_GATHER] = {"us_per_call": round(us, 2), "GBps": round(nb / us / 1e3, 1),
                                  "frac": round(nb / us / 1e3 / peak, 3), "copies": ncopy,
                                  "pages_GiBps_one_way": round(nb / 2 / us / 1e3 * 1e9 / 2 ** 30, 1)}
    del sets
    torch.cuda.empty_cache()
    _, _, tpeak = peaks()
    for name in prefill_configs():
        us, flops, nbytes, pcopies = time_prefill_workload(name, dev, ops)
        tf = flops / us / 1e6
        out["prefill"][name] = {"us_per_call": round(us, 2), "TFLOPs": round(tf, 1),
                                "frac_tensor": round(tf / tpeak, 3),
                                "GBps": round(nbytes / us / 1e3, 1), "copies": pcopies}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="pkd", choices=["pkd", "reference"])
    ap.add_argument("--no-targets", action="store_true", help="skip the side lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--sweep", action="store_true",
                    help="time every decode workload and gather point (one JSON line each)")
    ap.add_argument("--partition-size", type=int, default=0,
                    help="--sweep/--profile decode lines: forced partition_size "
                         "(0 = the library's plan, -1 = the stream form)")
    ap.add_argument("--tight-pool", action="store_true",
                    help="--profile decode: a pool of just the blocks the sequences use")
    ap.add_argument("--profile", default=None, metavar="KIND:NAME",
                    help="profiling mode: run only 'decode:<workload>', 'prefill:<workload>' or "
                         "'gather:<workload>' "
                         "warmup + steps times (no timing, no JSON line), e.g. under ncu")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.steps = max(args.steps, 1)

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        # Only rank 0 times the oracle; other ranks exit without work.
        return run_reference(args, world, rank)
    if args.profile:
        return run_profile(args, local)
    if args.sweep:
        return run_sweep(args, local)
    import torch

    from paged_kv_decode_22_gb300 import ops

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    peak, peak_src, _ = peaks()
    d = device_decode_inputs(HEADLINE, dev)
    S, H, D = d["q"].shape
    Hk, B = d["kc"].shape[2], d["kc"].shape[1]
    step_bytes = d["bytes"]
    ps, npart, path, ws_bytes = ops.decode_plan(S, H, Hk, D, B, d["max_ctx"])
    work = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        ops.paged_decode_attention(d["out"], d["q"], d["kc"], d["vc"], d["bt"], d["cl"],
                                   d["max_ctx"], d["scale"], workspace=work, stream=stream)

    # Warm-up, timed loosely to size the clock pre-roll.
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.warmup):
        call()
    barrier()
    warm_us = (time.perf_counter() - t0) * 1e6 / args.warmup
    preroll = preroll_calls(warm_us)
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with ClockSampler(gpu_id) as clocks:
        for _ in range(preroll):        # untimed: GPU under load while clocks are sampled
            call()
        barrier()
        timed_loop(call, args.steps, lambda i: ev[i].record(stream))
        barrier()
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    ms = max_over_ranks(ms, dist, dev)
    us = ms * 1e3

    # End to end through the public API with host buffers: every step copies
    # q, the block tables and the lengths in from pinned host memory, runs the
    # call and copies out back to pinned host memory.  The KV pool is resident
    # state, as in serving.  Steps are pipelined as a serving loop runs them:
    # two sets of device inputs and outputs, step i + 1's inputs come in on
    # one copy stream and step i's output goes out on another while a call
    # runs; each call waits for its own inputs, and each buffer set is reused
    # only after its call and its output copy are done.  The timed region
    # ends when the last output has reached the host.
    hq = d["q"].cpu().pin_memory()
    hbt = d["bt"].cpu().pin_memory()
    hcl = d["cl"].cpu().pin_memory()
    hout = [torch.empty(d["out"].shape, dtype=d["out"].dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hbt, hcl))
    d2h = hout[0].numel() * hout[0].element_size()
    bufs = [{k: d[k] for k in ("q", "bt", "cl", "out")},
            {k: torch.empty_like(d[k]) for k in ("q", "bt", "cl", "out")}]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer set b landed
    ev_call = [torch.cuda.Event() for _ in range(2)]   # call on buffer set b done
    ev_out = [torch.cuda.Event() for _ in range(2)]    # output of buffer set b on the host
    nstep = [0]

    def e2e_step():
        b = nstep[0] & 1
        nstep[0] += 1
        x = bufs[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_call[b])          # the previous call on this set has read its inputs
            x["q"].copy_(hq, non_blocking=True)
            x["bt"].copy_(hbt, non_blocking=True)
            x["cl"].copy_(hcl, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])             # this set's previous output has left
        ops.paged_decode_attention(x["out"], x["q"], d["kc"], d["vc"], x["bt"], x["cl"],
                                   d["max_ctx"], d["scale"], workspace=work, stream=stream)
        ev_call[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_call[b])
            hout[b].copy_(x["out"], non_blocking=True)
            ev_out[b].record(s_out)

    for _ in range(4):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    timed_loop(e2e_step, args.steps, lambda i: None)
    barrier()                                    # every stream, the last output copy included
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps, dist, dev)
    # The pipelined outputs are the same call's: check the last one.
    if not torch.equal(hout[(nstep[0] - 1) & 1], d["out"].cpu()):
        raise RuntimeError("pipelined end-to-end output differs from the device-timed call's")
    del d, work, bufs
    torch.cuda.empty_cache()

    sides = None
    if not args.no_targets:
        sides = side_lines(dev, ops, peak)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    achieved = step_bytes / us / 1e3
    traffic = stored_traffic(HEADLINE, DECODE_SOURCES)
    line = {
        "metric": METRIC, "value": round(whole_job_gbps(step_bytes, world, ms), 1),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "us_per_call": round(us, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 from a torch generator, random "
                "non-overlapping block tables)",
        "config": {"workload": HEADLINE, "shape": HEADLINE_DESC,
                   "l2": f"inputs larger than L2: {step_bytes / 1e9:.2f} GB of K/V per call "
                         "streamed through the 129 MB L2 (no flush needed)",
                   "decode_path": PATH_NAMES[path], "decode_partitions": npart,
                   "clock_preroll_calls": preroll},
        "step_bytes": step_bytes,
        "gpu_launches": decode_launches(npart, path) * args.steps,
        "roofline": {"kernel": "paged_decode_attention call (decode_tc_kernel + "
                               "stream_merge_kernel)" if path == 3 else
                               f"paged_decode_attention call ({PATH_NAMES[path]})",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 3),
                     "traffic": traffic, "algorithmic_bytes": step_bytes},
        "e2e": {"value": round(whole_job_gbps(step_bytes, world, e2e_ms), 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipelining": "two device buffer sets; each step's host copies run on two copy "
                              "streams beside the neighbouring steps' calls"},
        "clocks": clocks.summary(),
    }
    if sides is not None:
        line["side"] = sides
    if world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(HEADLINE)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
