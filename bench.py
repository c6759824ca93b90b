#!/usr/bin/env python3
"""Benchmark: paged decode attention + gather_cached_kv on one GB300.

One step is one pass of the whole hot path over one batch: a decode-attention
call (split-context partitions + log-sum-exp merge when the plan splits) and a
gather_cached_kv call.  Default workload: the LLaMA-13B-shaped MHA decode of
"Optimizes the single_query_cached_kv_attention kernel" (8 sequences x 40
heads, head_size 128, block_size 16, context 256, fp16, 2048-block pool) and
the largest point of the gather sweep of "Memcpy kernel for flash attention"
(2048 tokens, 40 heads, head_size 128, block_size 8, 1024 blocks, fp16).

Prints ONE JSON line (rank 0).  `value` is algorithmic HBM bytes per step
divided by device time per step (GB/s, 1e9).  Inputs rotate over enough
device copies that every step reads data not left in L2 by the last one.

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
# The CPU oracle legs run single-threaded; set before NumPy loads its BLAS.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

METRIC = ("paged decode attn µs/call and achieved HBM GB/s (% of GB300 roofline) "
          "vs oracle")
WORKLOAD = "llama13b_mha_b8_ctx256 decode + gather_t2048"
DECODE_CFG = "llama13b_mha_b8_ctx256"
GATHER_CFG = "gather_t2048"
# Decode workloads at batch >= 64 and context >= 1024, reported beside the
# default line (decode alone).
TARGETS = ["gqa_ctx1024_b64", "gqa_ctx1024_b256", "gqa_ctx4096_b64", "gqa_ctx4096_b256",
           "mqa_ragged_b64"]
PATH_NAMES = {0: "simt", 1: "tc", 2: "tc_cluster", 3: "tc_stream"}   # decode_plan's kernel family
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic per launch of the dominant kernel from an ncu capture, keyed by
# the sha256 (first 16 hex digits) of the kernel source it was taken on; the
# value is reported only while that source is unchanged.
NCU_TRAFFIC = {
    # gather_t2048, profiles/gather_cached_kv_t2048.md: 41.97 MB read + 1.80 MB
    # written during the kernel (its output is still dirty in L2 when it ends)
    "aba4662af3507d10": 41969152 + 1797376,
    # llama13b_mha_b8_ctx256, profiles/decode_simt_llama13b_mha_b8_ctx256.md
    "90c0e845acbd2fec": 42051328 + 56576,
}


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


def src_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


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


# ---------------------------------------------------------------- reference arm (oracle)

def _oracle_sample(c, g, n):
    """The first n units of the step: unit i = decode of (sequence i // H, head
    i % H) over its whole context plus gather of 16 tokens."""
    from oracle.gather import gather_cached_kv as ref_gather
    from oracle.paged_attention import paged_decode_attention as ref_attn
    H = c.num_heads
    pairs = [(i // H, i % H) for i in range(n)]
    tokens = g.slot_mapping[: min(g.num_tokens, 16 * n)]
    per_pair = decode_bytes(c) / (c.num_seqs * H)
    nbytes = per_pair * n + gather_bytes(g) * len(tokens) / g.num_tokens

    def run():
        ref_attn(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens, c.scale,
                 c.dtype, pairs=pairs)
        ref_gather(g.key_cache, g.value_cache, tokens)
    return run, nbytes, f"decode (seq, head) pairs 0..{n - 1} of {c.num_seqs * H} + " \
                        f"gather tokens 0..{len(tokens) - 1} of {g.num_tokens}"


def run_reference(args, world, rank):
    """The oracle as it stands, timed on the host cores, as the reference arm."""
    if rank != 0:
        return 0
    from paged_kv_decode_22_gb300.workloads import (decode_configs, gather_sweep,
                                                    make_decode_case, make_gather_case)
    c = make_decode_case(name=DECODE_CFG, **decode_configs()[DECODE_CFG])
    g = make_gather_case(name=GATHER_CFG, **gather_sweep()[GATHER_CFG])
    full = c.num_seqs * c.num_heads
    # Size the per-step sample so that warm-up + timed steps take about 60 s.
    run1, _, _ = _oracle_sample(c, g, 1)
    t0 = time.perf_counter()
    for _ in range(5):
        run1()
    t_unit = (time.perf_counter() - t0) / 5
    n = int(max(1, min(full, 60.0 / max(1, args.steps + args.warmup) / t_unit)))
    run, nbytes, what = _oracle_sample(c, g, n)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) fp16 inputs, random non-overlapping block tables)",
        "config": {"workload": WORKLOAD, "sample": what},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": what},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def cpu_baseline(c, g, budget_s=10.0):
    """The oracle as it stands on the host, on a bounded sample of the step."""
    run, nbytes, what = _oracle_sample(c, g, 16)
    n, t0 = 0, time.perf_counter()
    while True:
        run()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(nbytes * n / el / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "sample": f"{what}; {n} passes in {el:.1f} s"}


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


def device_decode_inputs(name, dev):
    """Device inputs of a decode workload from a seeded torch generator (for
    timing and profiling: the kernels' speed does not depend on the values)."""
    import torch

    from paged_kv_decode_22_gb300.workloads import decode_configs
    cfg = decode_configs()[name]
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg["seed"])
    S, H, Hk, D, B = (cfg["num_seqs"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_size"],
                      cfg["block_size"])
    lens = torch.tensor(cfg["context_lens"], dtype=torch.int32)
    need = (lens + B - 1) // B
    nb = max(cfg["num_blocks"], int(need.sum()))
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
        d = device_decode_inputs(name, dev)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="pkd", choices=["pkd", "reference"])
    ap.add_argument("--no-targets", action="store_true", help="skip the large-batch GQA lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--sweep", action="store_true",
                    help="time every decode workload and gather point (one JSON line each)")
    ap.add_argument("--partition-size", type=int, default=0,
                    help="--sweep/--profile decode lines: forced partition_size "
                         "(0 = the library's plan, -1 = the stream form)")
    ap.add_argument("--profile", default=None, metavar="KIND:NAME",
                    help="profiling mode: run only 'decode:<workload>', 'prefill:<workload>' or "
                         "'gather:<workload>' "
                         "warmup + steps times (no timing, no JSON line), e.g. under ncu")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

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
    import numpy as np
    import torch

    from paged_kv_decode_22_gb300 import ops
    from paged_kv_decode_22_gb300.workloads import (decode_configs, gather_sweep,
                                                    make_decode_case, make_gather_case)

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

    c = make_decode_case(name=DECODE_CFG, **decode_configs()[DECODE_CFG])
    g = make_gather_case(name=GATHER_CFG, **gather_sweep()[GATHER_CFG])
    f16 = torch.float16

    def upd(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                             else np.ascontiguousarray(a))
        return (t.view(dt) if dt is not None else t).to(dev)

    step_bytes = decode_bytes(c) + gather_bytes(g)
    # Rotation: enough independent device copies of every input and output
    # that consecutive steps never find their data in L2 (touched bytes x
    # copies > 3 x L2).
    ncopy = max(2, math.ceil(3 * L2_BYTES / step_bytes))
    sets = []
    for _ in range(ncopy):
        sets.append(dict(q=upd(c.q, f16), kc=upd(c.key_cache, f16), vc=upd(c.value_cache, f16),
                         bt=upd(c.block_tables), cl=upd(c.context_lens),
                         gkc=upd(g.key_cache, f16), gvc=upd(g.value_cache, f16),
                         slots=upd(g.slot_mapping),
                         out=torch.empty(c.q.shape, dtype=f16, device=dev),
                         ko=torch.empty((g.num_tokens, g.num_heads, g.head_size), dtype=f16,
                                        device=dev),
                         vo=torch.empty((g.num_tokens, g.num_heads, g.head_size), dtype=f16,
                                        device=dev)))
    S, H, D = c.q.shape
    ps, npart, path, ws_bytes = ops.decode_plan(S, H, c.num_kv_heads, D, c.block_size,
                                                c.max_context_len)
    work = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def decode_call(i, st=None):
        d = sets[i % ncopy]
        ops.paged_decode_attention(d["out"], d["q"], d["kc"], d["vc"], d["bt"], d["cl"],
                                   c.max_context_len, c.scale, workspace=work, stream=st)

    def gather_call(i, st=None):
        d = sets[i % ncopy]
        ops.gather_cached_kv(d["ko"], d["vo"], d["gkc"], d["gvc"], d["slots"], stream=st)

    launches_per_step = 2 + (1 if npart > 1 else 0)
    for i in range(args.warmup):
        decode_call(i, stream)
        gather_call(i, stream)
    barrier()

    # The timed steps replay CUDA graphs of CHUNK decode calls followed by CHUNK
    # gather calls (inputs rotating over the device copies), so host launch
    # overhead stays out of the device time.  Events between the two graphs
    # give each kernel's average duration inside the same timed region.
    CHUNK = 64

    def capture(fn, n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(n):
                fn(i)
        return gr

    full, rest = divmod(args.steps, CHUNK)
    graphs = [(capture(decode_call, CHUNK), capture(gather_call, CHUNK))] if full else []
    tail = (capture(decode_call, rest), capture(gather_call, rest)) if rest else None
    plan = [graphs[0]] * full + ([tail] if tail else [])
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    for gd, gg in plan[:2]:
        gd.replay()
        gg.replay()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(plan) + 1)]
    with ClockSampler(gpu_id) as clocks:
        barrier()
        evs[0].record(stream)
        for j, (gd, gg) in enumerate(plan):
            gd.replay()
            evs[2 * j + 1].record(stream)
            gg.replay()
            evs[2 * j + 2].record(stream)
        barrier()
    total_ms = evs[0].elapsed_time(evs[-1])
    dec_ms = sum(evs[2 * j].elapsed_time(evs[2 * j + 1]) for j in range(len(plan)))
    gat_ms = sum(evs[2 * j + 1].elapsed_time(evs[2 * j + 2]) for j in range(len(plan)))
    ms = total_ms / args.steps
    ms = max_over_ranks(ms, dist, dev)
    dec_us = dec_ms * 1e3 / args.steps
    gat_us = gat_ms * 1e3 / args.steps
    del graphs, tail, plan

    # End to end through the public API with host buffers: per step, copy the
    # step's inputs (q, block tables, context lengths, slot mapping) from
    # pinned host memory, run both calls, read every output back to pinned host
    # memory.  The KV pools are resident state, as in serving.
    hq = torch.from_numpy(c.q.view(np.int16)).view(f16).pin_memory()
    hbt = torch.from_numpy(c.block_tables).pin_memory()
    hcl = torch.from_numpy(c.context_lens).pin_memory()
    hsl = torch.from_numpy(g.slot_mapping).pin_memory()
    hout = torch.empty(sets[0]["out"].shape, dtype=f16).pin_memory()
    hko = torch.empty(sets[0]["ko"].shape, dtype=f16).pin_memory()
    hvo = torch.empty(sets[0]["vo"].shape, dtype=f16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hbt, hcl, hsl))
    d2h = sum(t.numel() * t.element_size() for t in (hout, hko, hvo))

    def e2e_step(i):
        d = sets[i % ncopy]
        d["q"].copy_(hq, non_blocking=True)
        d["bt"].copy_(hbt, non_blocking=True)
        d["cl"].copy_(hcl, non_blocking=True)
        d["slots"].copy_(hsl, non_blocking=True)
        decode_call(i, stream)
        gather_call(i, stream)
        hout.copy_(d["out"], non_blocking=True)
        hko.copy_(d["ko"], non_blocking=True)
        hvo.copy_(d["vo"], non_blocking=True)
        stream.synchronize()

    e2e_steps = max(20, min(2000, args.steps // 10))
    for i in range(5):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    barrier()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps

    # Large-batch decode lines (decode alone): inputs from a seeded torch
    # generator on the device (timing does not depend on the values), CUDA
    # graph replays over rotated copies, as in the timed region above.
    targets = {}
    if not args.no_targets:
        for name in TARGETS:
            us, nbytes, (ps, npx, pathx, _), tcopies = time_decode_workload(name, dev, ops)
            targets[name] = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                             "path": PATH_NAMES[pathx], "partitions": npx,
                             "copies": tcopies}

    # Prefill lines (tensor-bound): same method, FLOPs against the bf16 peak.
    prefill_lines = {}
    if not args.no_targets:
        from paged_kv_decode_22_gb300.workloads import prefill_configs
        for name in prefill_configs():
            us, flops, nbytes, pcopies = time_prefill_workload(name, dev, ops)
            prefill_lines[name] = {"us_per_call": round(us, 2), "TFLOPs": round(flops / us / 1e6, 1),
                                   "GBps": round(nbytes / us / 1e3, 1), "copies": pcopies}

    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    tpeak = FALLBACK_BF16_TFLOPS
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            pk = json.load(f)
        if pk.get("hbm_gbs"):
            peak, peak_src = float(pk["hbm_gbs"]), "measured"
        if pk.get("bf16_tflops"):
            tpeak = float(pk["bf16_tflops"])
    for v in targets.values():
        v["frac"] = round(v["GBps"] / peak, 3)
    for v in prefill_lines.values():
        v["frac_tensor"] = round(v["TFLOPs"] / tpeak, 3)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    dec_b, gat_b = decode_bytes(c), gather_bytes(g)
    if dec_us >= gat_us:
        dom, dom_bytes, dom_us, dom_src = "decode", dec_b, dec_us, ("paged_kv_decode_22_gb300/csrc/decode_simt.cu",)
    else:
        dom, dom_bytes, dom_us, dom_src = "gather_cached_kv", gat_b, gat_us, ("paged_kv_decode_22_gb300/csrc/copy_kv.cu",)
    achieved = dom_bytes / dom_us / 1e3
    traffic = NCU_TRAFFIC.get(src_hash(*dom_src))
    value = whole_job_gbps(step_bytes, world, ms)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic (seeded N(0,1) fp16, random non-overlapping block tables)",
        "config": {"workload": WORKLOAD, "decode": "S=8 H=40 Hk=40 D=128 B=16 ctx=256 NB=2048",
                   "gather": "T=2048 H=40 D=128 B=8 NB=1024",
                   "l2": f"inputs rotate over {ncopy} device copies (>3x L2 touched per cycle)",
                   "decode_partitions": npart, "decode_path": PATH_NAMES[path]},
        "decode_us_per_call": round(dec_us, 2), "gather_us_per_call": round(gat_us, 2),
        "step_bytes": step_bytes,
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "traffic": traffic,
                     "algorithmic_bytes": dom_bytes},
        "e2e": {"value": round(step_bytes / e2e_ms / 1e6, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clocks.summary(),
        "targets_decode": targets,
        "targets_prefill": prefill_lines,
    }
    if world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(c, g)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
