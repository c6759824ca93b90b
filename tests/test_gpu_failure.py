"""Failure detection without a GPU fault: a bounded wait that nothing
satisfies gives up, reports PKD_DEV_TIMEOUT through the status word, and
leaves the context usable (a decode call afterwards still matches the
oracle)."""
import ctypes
import time

import pytest
import torch

from oracle.paged_attention import paged_decode_attention as oracle_attention
from paged_kv_decode_22_gb300 import _lib
from paged_kv_decode_22_gb300.workloads import make_decode_case

from .gpu_util import DeviceCase, assert_close, run_decode

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    limit_ns = 20_000_000                      # 20 ms
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = _lib.lib().pkd_selftest_bounded_wait(ctypes.c_void_p(status.data_ptr()), limit_ns,
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == _lib.DEV_TIMEOUT
    assert elapsed >= limit_ns * 1e-9 * 0.9     # the wait really waited
    assert elapsed < 5.0                        # and then gave up
    c = make_decode_case(seed=151, num_seqs=3, num_heads=32, num_kv_heads=4, head_size=128,
                         block_size=16, num_blocks=64, context_lens=[300, 1, 129], dtype="bf16")
    got, st2 = run_decode(DeviceCase(c))
    assert st2 == 0
    assert_close(got, oracle_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                       c.context_lens, c.scale, c.dtype), "decode after a time-out")
