"""Concurrent first calls from several host threads, in a fresh process.

The launch code keeps per-device host state that the first call of each
kernel sets: shared-memory size attributes, cluster capacities, device
attributes.  Seven threads make their first calls together, each on its
own stream and each through a different kernel.  The kernels are CUDA-core
decode, tensor-core decode, stream form, cluster form, prefill, and
bulk and 16-byte gathers.  Every output and status word must equal, bit for
bit, the same call made afterwards with no other call running.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import threading
import numpy as np
import torch
from paged_kv_decode_22_gb300 import ops
from paged_kv_decode_22_gb300.workloads import make_decode_case, make_gather_case, make_prefill_case
from tests.gpu_util import TORCH_DT, down_bits, up


def decode_job(seed, H, Hk, lens, dtype, ps, path):
    need = sum(-(-L // 16) for L in lens)
    c = make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk, head_size=128,
                         block_size=16, num_blocks=need + 4, context_lens=lens, dtype=dtype)
    plans.append((len(lens), H, Hk, c.max_context_len, ps, path))
    args = (up(c.q, dtype), up(c.key_cache, dtype), up(c.value_cache, dtype), up(c.block_tables),
            up(c.context_lens))

    def run(stream):
        with torch.cuda.stream(stream):
            out = torch.zeros(c.q.shape, dtype=TORCH_DT[dtype], device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            ops.paged_decode_attention(out, *args, c.max_context_len, c.scale, partition_size=ps,
                                       device_status=st, stream=stream)
        stream.synchronize()
        return down_bits(out), int(st.item())
    return run


def prefill_job(seed, chunks):
    lens = [L for L, _ in chunks]
    need = sum(-(-L // 16) for L in lens)
    c = make_prefill_case(seed=seed, num_seqs=len(chunks), num_heads=64, num_kv_heads=8,
                          head_size=128, block_size=16, num_blocks=need + 4, context_lens=lens,
                          query_lens=[n for _, n in chunks], dtype="bf16")
    b = c.base
    args = (up(c.q, "bf16"), up(b.key_cache, "bf16"), up(b.value_cache, "bf16"),
            up(b.block_tables), up(b.context_lens), up(c.query_start))

    def run(stream):
        with torch.cuda.stream(stream):
            out = torch.zeros(c.q.shape, dtype=torch.bfloat16, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            ops.paged_prefill_attention(out, *args, int(c.query_lens.max()), b.max_context_len,
                                        b.scale, device_status=st, stream=stream)
        stream.synchronize()
        return down_bits(out), int(st.item())
    return run


def gather_job(seed, T):
    g = make_gather_case(seed=seed, num_tokens=T, num_heads=40, head_size=128, block_size=8,
                         num_blocks=160, dtype="fp16")
    args = (up(g.key_cache, "fp16"), up(g.value_cache, "fp16"), up(g.slot_mapping))

    def run(stream):
        with torch.cuda.stream(stream):
            ko = torch.zeros((T, 40, 128), dtype=torch.float16, device="cuda")
            vo = torch.zeros_like(ko)
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            ops.gather_cached_kv(ko, vo, *args, device_status=st, stream=stream)
        stream.synchronize()
        return np.concatenate([down_bits(ko), down_bits(vo)]), int(st.item())
    return run


plans = []   # checked after the concurrent calls, so that those are the first
rng = np.random.default_rng(5)
jobs = [
    decode_job(1, 40, 40, [256] * 8, "fp16", 0, ops.PATH_SIMT),
    decode_job(2, 64, 8, [1024] * 16, "bf16", 0, ops.PATH_TC),
    decode_job(3, 48, 1, [int(x) for x in rng.integers(1, 2000, 40)], "fp16", ops.PARTITION_STREAM,
               ops.PATH_TC_STREAM),
    decode_job(4, 64, 8, [4096], "bf16", 0, ops.PATH_TC_CLUSTER),
    prefill_job(6, [(1000, 256), (600, 256)]),
    gather_job(7, 100),
    gather_job(8, 1200),
]
torch.cuda.synchronize()
streams = [torch.cuda.Stream() for _ in jobs]
results = [None] * len(jobs)
gate = threading.Barrier(len(jobs))


def worker(i):
    gate.wait()
    results[i] = jobs[i](streams[i])


threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
for t in threads:
    t.start()
for t in threads:
    t.join()
for i, job in enumerate(jobs):
    bits, st = job(torch.cuda.current_stream())
    assert results[i] is not None, i
    assert results[i][1] == st == 0, (i, results[i][1], st)
    assert np.array_equal(results[i][0], bits), i
for S, H, Hk, L, ps, path in plans:
    assert ops.decode_plan(S, H, Hk, 128, 16, L, ps)[2] == path, (S, H, Hk, L, ps, path)
print("ok")
'''


def test_concurrent_first_calls_from_host_threads():
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.strip().endswith("ok"), r.stdout[-2000:]
