"""Decode attention on the GPU (through the C ABI) against the CPU oracle.

Tolerance: max |gpu - oracle| <= 1e-2 and mean <= 1e-3 over the compared
elements, outputs decoded from fp16/bf16 and the oracle in float64.
"""
import functools

import numpy as np
import pytest
import torch

from oracle.formats import decode_bits
from oracle.paged_attention import paged_decode_attention as oracle_attention
from paged_kv_decode_22_gb300.workloads import decode_configs, make_decode_case

from .gpu_util import DeviceCase, assert_close, run_decode, up

pytestmark = pytest.mark.gpu

SMALL = ["tiny_mha", "llama13b_mha_b8_ctx256", "gqa_ctx1024_b1", "gqa_ctx1024_b4",
         "gqa_ctx4096_b1", "gqa_ctx4096_bs256_b1", "gqa_ctx1024_b16"]
LARGE = ["gqa_ctx1024_b64", "gqa_ctx1024_b256", "gqa_ctx4096_b16", "gqa_ctx4096_b64",
         "gqa_ctx4096_b256", "gqa_ctx4096_bs256_b256", "mqa_ragged_b64"]


@functools.lru_cache(maxsize=2)
def _device_case(name):
    return DeviceCase(make_decode_case(name=name, **decode_configs()[name]))


def _oracle(c, pairs=None, **kw):
    return oracle_attention(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens,
                            c.scale, c.dtype, pairs=pairs, **kw)


@pytest.mark.parametrize("name", SMALL)
def test_workload_parity_full(name):
    dc = _device_case(name)
    got, status = run_decode(dc)
    assert status == 0
    assert_close(got, _oracle(dc.c), name)


@pytest.mark.parametrize("name", LARGE)
def test_workload_parity_full_size(name):
    # Every (sequence, head) row at full size, in the launch configuration the
    # bench times (the library's own plan): the stream form's cut pairs and
    # their merges at every range edge are all compared.
    from paged_kv_decode_22_gb300 import ops
    dc = _device_case(name)
    c = dc.c
    plan = ops.decode_plan(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_size, c.block_size,
                           c.max_context_len)
    got, status = run_decode(dc)
    assert status == 0
    assert np.isfinite(got).all()
    assert_close(got, _oracle(c), f"{name}, plan {plan}")


@pytest.mark.parametrize("partition_size", [64, 128, 192, 512, 4096])
def test_partition_count_does_not_change_the_result(partition_size):
    dc = _device_case("gqa_ctx4096_b1")
    base, _ = run_decode(dc, partition_size=4096)
    got, status = run_decode(dc, partition_size=partition_size)
    assert status == 0
    assert_close(got, _oracle(dc.c), f"partition {partition_size}")
    assert np.abs(got - base).max() <= 2e-2


def _ragged(seed, H, Hk, D, B, lens, dtype, nb=None):
    need = sum(-(-L // B) for L in lens)
    return make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                            head_size=D, block_size=B, num_blocks=nb or need + 7,
                            context_lens=lens, dtype=dtype)


RAGGED = [
    # (H, Hk, D, B, dtype): group sizes 1, 2, 3, 4, 8, 48; both head sizes; block sizes 8..256
    (8, 8, 128, 16, "fp16"), (8, 4, 128, 8, "bf16"), (12, 4, 64, 32, "fp16"),
    (16, 4, 128, 64, "bf16"), (64, 8, 128, 16, "bf16"), (48, 1, 128, 16, "fp16"),
    (16, 2, 64, 128, "bf16"), (8, 1, 128, 256, "fp16"), (4, 4, 64, 16, "bf16"),
    (32, 1, 128, 16, "bf16"), (64, 1, 128, 32, "fp16"), (40, 8, 128, 16, "bf16"),
]


@pytest.mark.parametrize("H,Hk,D,B,dtype", RAGGED)
@pytest.mark.parametrize("partition_size", [0, 64, 128])
def test_ragged_lengths_and_edges(H, Hk, D, B, dtype, partition_size):
    lens = [1, B - 1, B, B + 1, 63, 64, 65, 127, 128, 129, 0, 300, 2 * B + 3]
    c = _ragged(17, H, Hk, D, B, lens, dtype)
    dc = DeviceCase(c)
    got, status = run_decode(dc, partition_size=partition_size)
    assert status == 0
    assert_close(got, _oracle(c), f"H{H}/{Hk} D{D} B{B} {dtype} ps{partition_size}")
    assert (got[lens.index(0)] == 0).all()


@pytest.mark.parametrize("H,Hk,dtype", [(32, 4, "bf16"), (48, 1, "fp16"), (8, 8, "fp16")])
@pytest.mark.parametrize("partition_size", [0, 64])
def test_more_sequences_than_the_schedule_table_holds(H, Hk, dtype, partition_size):
    # 1100 sequences: past the 1024 whose lengths the kernels keep in shared
    # memory, units are dealt round-robin from lengths read in global memory
    # (tensor-core groups), and the stream form is not offered.
    from paged_kv_decode_22_gb300 import ops
    lens = [int(L) for L in np.random.default_rng(41).integers(0, 200, 1100)]
    c = _ragged(43, H, Hk, 128, 16, lens, dtype)
    _, npart, path, _ = ops.decode_plan(c.num_seqs, H, Hk, 128, 16, c.max_context_len,
                                        partition_size)
    assert path != ops.PATH_TC_STREAM
    got, status = run_decode(DeviceCase(c), partition_size=partition_size)
    assert status == 0
    assert_close(got, _oracle(c), f"1100 sequences H{H}/{Hk} {dtype} ps{partition_size} path {path}")
    assert (got[np.asarray(lens) == 0] == 0).all()


ALIBI = [(8, 8, 128, 16, "fp16"), (12, 4, 64, 32, "bf16"), (64, 8, 128, 16, "bf16"),
         (48, 1, 128, 16, "fp16"), (32, 1, 128, 64, "bf16")]


@pytest.mark.parametrize("H,Hk,D,B,dtype", ALIBI)
@pytest.mark.parametrize("partition_size", [0, 128])
def test_alibi_matches_oracle(H, Hk, D, B, dtype, partition_size):
    from paged_kv_decode_22_gb300 import ops

    from .gpu_util import down_bits
    lens = [1, B + 1, 300, 127, 1000, 0]
    c = _ragged(23, H, Hk, D, B, lens, dtype)
    dc = DeviceCase(c)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32)
    out = torch.full(c.q.shape, float("nan"), dtype=dc.q.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, c.max_context_len,
                               c.scale, partition_size=partition_size, device_status=status,
                               alibi_slopes=torch.from_numpy(slopes).cuda())
    torch.cuda.synchronize()
    got = decode_bits(down_bits(out), dtype)
    ref = _oracle(c, alibi_slopes=slopes.astype(np.float64))
    assert int(status.item()) == 0
    assert_close(got, ref, f"alibi H{H}/{Hk} D{D} B{B} ps{partition_size}")
    # Slopes of zero reproduce plain attention.
    ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, c.max_context_len,
                               c.scale, partition_size=partition_size,
                               alibi_slopes=torch.zeros(H, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert_close(decode_bits(down_bits(out), dtype), _oracle(c), "zero slopes")


def test_single_token_returns_value_row_exactly():
    c = _ragged(3, 16, 2, 128, 16, [1, 1, 1], "bf16")
    got, _ = run_decode(DeviceCase(c))
    for s in range(3):
        for h in range(16):
            v = decode_bits(c.value_cache[c.block_tables[s, 0], 0, h // 8], "bf16")
            np.testing.assert_array_equal(got[s, h], v)


def test_block_permutation_invariance():
    c = _ragged(5, 32, 4, 128, 16, [77, 500, 1000], "fp16", nb=200)
    a, _ = run_decode(DeviceCase(c))
    perm = np.random.default_rng(9).permutation(c.num_blocks)
    inv = np.argsort(perm)
    c.key_cache = c.key_cache[perm]
    c.value_cache = c.value_cache[perm]
    c.block_tables = np.where(c.block_tables >= 0, inv[np.maximum(c.block_tables, 0)],
                              -1).astype(np.int32)
    b, _ = run_decode(DeviceCase(c))
    assert np.abs(a - b).max() <= 1e-6


def test_bad_block_and_bad_length_set_status_and_zero_rows():
    c = _ragged(11, 8, 2, 128, 16, [40, 40, 40, 40, 40], "bf16", nb=40)
    dc = DeviceCase(c)
    bt = c.block_tables.copy()
    bt[1, 2] = c.num_blocks + 3          # id past the pool
    bt[3, 0] = -5                        # negative id
    got, status = run_decode(dc, block_tables=up(bt))
    assert status & 1
    assert (got[1] == 0).all() and (got[3] == 0).all()
    ref = _oracle(c)
    for s in (0, 2, 4):
        assert_close(got[s], ref[s], f"seq {s}")

    lens = c.context_lens.copy()
    lens[0] = -1
    lens[2] = 41                         # longer than max_context_len given below
    lens[4] = bt.shape[1] * 16 + 1       # longer than the block table
    for ps in (0, 64):
        got, status = run_decode(dc, context_lens=up(lens), max_context_len=40,
                                 partition_size=ps)
        assert status & 4
        for s in (0, 2, 4):
            assert (got[s] == 0).all()
        for s in (1, 3):
            assert_close(got[s], ref[s], f"seq {s}")


def test_workspace_bytes_covers_every_plan_of_its_sizes():
    from paged_kv_decode_22_gb300 import ops
    for S, H, D, ctx in [(1, 64, 128, 4096), (4, 64, 128, 1024), (64, 48, 128, 8192),
                         (8, 40, 128, 256), (256, 64, 128, 4096), (2, 4, 64, 40)]:
        w = ops.decode_workspace_bytes(S, H, D, ctx)
        need = [ops.decode_plan(S, H, hk, D, b, ctx)[3] for hk in range(1, H + 1) if H % hk == 0
                for b in (8, 16, 32, 64, 128, 256)]
        assert w == max(need), (S, H, D, ctx)
    # A call with a workspace of exactly that size.
    c = _ragged(29, 64, 8, 128, 16, [4096, 1, 2000, 3333], "bf16")
    dc = DeviceCase(c)
    w = ops.decode_workspace_bytes(4, 64, 128, c.max_context_len)
    assert w > 0
    work = torch.empty(w, dtype=torch.uint8, device="cuda")
    out = torch.empty(c.q.shape, dtype=torch.bfloat16, device="cuda")
    ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, c.max_context_len, c.scale,
                               workspace=work)
    torch.cuda.synchronize()
    from .gpu_util import down_bits
    assert_close(decode_bits(down_bits(out), "bf16"), _oracle(c), "workspace_bytes-sized workspace")


def test_workspace_too_small_is_rejected():
    from paged_kv_decode_22_gb300 import ops
    dc = _device_case("gqa_ctx4096_b1")
    c = dc.c
    ps, npart, _, ws = ops.decode_plan(1, 64, 8, 128, 16, 4096, 128)
    assert npart == 32 and ws > 0
    out = torch.empty(c.q.shape, dtype=torch.bfloat16, device="cuda")
    small = torch.empty(ws - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.PkdError) as e:
        ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, 4096, c.scale,
                                   partition_size=128, workspace=small)
    assert e.value.status == 4
    big = torch.empty(ws + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.PkdError) as e:
        ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, 4096, c.scale,
                                   partition_size=128, workspace=big[16:])
    assert e.value.status == 5


def test_runs_on_a_side_stream_and_in_a_cuda_graph():
    from paged_kv_decode_22_gb300 import ops
    dc = _device_case("gqa_ctx1024_b4")
    c = dc.c
    ref = _oracle(c)
    _, npart, _, ws = ops.decode_plan(4, 64, 8, 128, 16, 1024, 0)
    work = torch.empty(max(ws, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty(c.q.shape, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, 1024, c.scale,
                                   workspace=work)
    s.synchronize()
    from .gpu_util import down_bits
    assert_close(decode_bits(down_bits(out), "bf16"), ref, "side stream")
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, 1024, c.scale,
                                   workspace=work)
    g.replay()
    torch.cuda.synchronize()
    assert_close(decode_bits(down_bits(out), "bf16"), ref, "graph replay")
