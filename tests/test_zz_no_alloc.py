"""Allocation-free decode entry point (pkd_paged_decode_attention_static_ws).

It exists for callers that cannot allocate device memory while they run; its
split-context scratch is an array built into the library.  This file is
collected last so that a failure here cannot hide the other tests.  The test
calls the entry point through the C ABI twice in a row, on different inputs,
and checks each output against the ordinary entry point (caller-provided
workspace) and against the float64 oracle, within the decode tolerance; it
also checks that a plan needing more scratch than the built-in array is
refused before any launch.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle.formats import decode_bits
from oracle.paged_attention import paged_decode_attention as attn_ref
from paged_kv_decode_22_gb300 import _lib, ops
from paged_kv_decode_22_gb300.workloads import make_decode_case

from .gpu_util import ATOL_MAX, ATOL_MEAN, DeviceCase, assert_close, down_bits

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 * 1024 * 1024


def _static_call(dc, out, partition_size, status):
    c = dc.c
    return _lib.lib().pkd_paged_decode_attention_static_ws(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(dc.q.data_ptr()),
        ctypes.c_void_p(dc.kc.data_ptr()), ctypes.c_void_p(dc.vc.data_ptr()),
        ctypes.c_void_p(dc.bt.data_ptr()), c.max_blocks_per_seq,
        ctypes.c_void_p(dc.cl.data_ptr()), c.max_context_len, c.num_seqs, c.num_heads,
        c.num_kv_heads, c.head_size, c.block_size, c.num_blocks, ctypes.c_float(c.scale),
        1 if c.dtype == "bf16" else 0, partition_size, ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _case(seed, lens, H, Hk, dtype):
    need = sum(-(-L // 16) for L in lens)
    return DeviceCase(make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H,
                                       num_kv_heads=Hk, head_size=128, block_size=16,
                                       num_blocks=need + 5, context_lens=lens, dtype=dtype))


@pytest.mark.parametrize("partition_size", [128, 0, -1])
def test_static_scratch_entry_matches_ordinary_entry_twice(partition_size):
    # -1: the stream form (tensor-core shapes only); its scratch holds two
    # partial slots per SM and the range-edge descriptors.
    cases = [_case(31, [4096, 777], 64, 8, "bf16"),
             _case(32, [3000, 129, 2048], 16, 16, "fp16") if partition_size >= 0
             else _case(34, [5000, 1, 0, 3333], 48, 1, "fp16")]
    paths = []
    for dc in cases:                         # two calls in a row, different inputs
        c = dc.c
        _, npart, path, ws_bytes = ops.decode_plan(c.num_seqs, c.num_heads, c.num_kv_heads, 128,
                                                   16, c.max_context_len, partition_size)
        assert ws_bytes <= STATIC_BYTES
        paths.append((path, npart, ws_bytes))
        dt = torch.bfloat16 if c.dtype == "bf16" else torch.float16
        ref = torch.full(c.q.shape, float("nan"), dtype=dt, device="cuda")
        ops.paged_decode_attention(ref, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, c.max_context_len,
                                   c.scale, partition_size=partition_size)
        out = torch.full(c.q.shape, float("nan"), dtype=dt, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _static_call(dc, out, partition_size, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = decode_bits(down_bits(out), c.dtype)
        want = decode_bits(down_bits(ref), c.dtype)
        assert np.isfinite(got).all()
        err = np.abs(got - want)
        assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (err.max(), err.mean())
        assert_close(got, attn_ref(c.q, c.key_cache, c.value_cache, c.block_tables,
                                   c.context_lens, c.scale, c.dtype),
                     f"static scratch, plan (path, partitions, scratch bytes) {paths[-1]}")


def test_static_scratch_entry_refuses_plans_larger_than_its_array():
    dc = _case(33, [4096] * 4, 64, 8, "bf16")
    c = dc.c
    # A forced partition of 128 tokens over a claimed 256K-token context needs
    # 4 * 64 * 2048 * 130 * 4 bytes of scratch, far above the built-in array.
    big_ctx = 262144
    _, npart, _, ws_bytes = ops.decode_plan(4, 64, 8, 128, 16, big_ctx, 128)
    assert ws_bytes > STATIC_BYTES
    out = torch.zeros(c.q.shape, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = _lib.lib().pkd_paged_decode_attention_static_ws(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(dc.q.data_ptr()),
        ctypes.c_void_p(dc.kc.data_ptr()), ctypes.c_void_p(dc.vc.data_ptr()),
        ctypes.c_void_p(dc.bt.data_ptr()), c.max_blocks_per_seq,
        ctypes.c_void_p(dc.cl.data_ptr()), big_ctx, 4, 64, 8, 128, 16, c.num_blocks,
        ctypes.c_float(c.scale), 1, 128, ctypes.c_void_p(status.data_ptr()), None)
    assert st == 4                            # PKD_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bool((out == 0).all())
