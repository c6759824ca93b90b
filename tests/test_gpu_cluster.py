"""Split context merged inside thread-block clusters (PKD_PATH_TC_CLUSTER).

The partitions of one (sequence, KV head) run as one cluster and are merged
through distributed shared memory in the same launch.  Each case checks
through decode_plan that the cluster form is the one that runs, and compares
it with the float64 oracle (max |err| <= 1e-2, mean <= 1e-3) and with the
workspace form of the same split (forced by a larger max_context_len, which
raises the partition count past the cluster limit of 16).
"""
import numpy as np
import pytest
import torch

from oracle.formats import decode_bits
from oracle.paged_attention import paged_decode_attention as oracle_attention
from paged_kv_decode_22_gb300.workloads import make_decode_case

from .gpu_util import DeviceCase, assert_close, down_bits, run_decode, up

pytestmark = pytest.mark.gpu

# (H, Hk, D, B, dtype): group sizes 4..64, padded groups 16/32/48/64, block sizes 16..256
LAYOUTS = [(64, 8, 128, 16, "bf16"), (48, 1, 128, 16, "fp16"), (16, 4, 128, 64, "bf16"),
           (40, 1, 128, 32, "fp16"), (48, 4, 128, 16, "bf16"), (32, 1, 128, 128, "bf16"),
           (4, 1, 128, 256, "fp16"), (24, 2, 128, 16, "fp16")]


def _case(seed, H, Hk, D, B, lens, dtype):
    need = sum(-(-L // B) for L in lens)
    return make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                            head_size=D, block_size=B, num_blocks=need + 5, context_lens=lens,
                            dtype=dtype)


def _lens(Hk, ps, P):
    """Ragged lengths for a split into P partitions of ps tokens: the full
    span, a length that ends inside the first partition (so later ranks of
    its cluster are empty), one past a partition boundary, a single token and
    zero; as many sequences as keep S * Hk clusters small."""
    span = P * ps
    pool = [span, ps - 5, ps + 1, span - 37, 1, 0, 2 * ps, span - ps + 3]
    n = max(1, min(len(pool), 64 // (Hk * P)))
    return pool[:n] if n > 1 else [span - 11]


def _plan(c, ps, max_ctx=None):
    from paged_kv_decode_22_gb300 import ops
    return ops.decode_plan(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_size, c.block_size,
                           max_ctx or c.max_context_len, ps)


def _oracle(c, **kw):
    return oracle_attention(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens,
                            c.scale, c.dtype, **kw)


@pytest.mark.parametrize("H,Hk,D,B,dtype", LAYOUTS)
@pytest.mark.parametrize("ps,P", [(128, 2), (256, 4), (128, 8), (128, 16)])
def test_cluster_merge_matches_oracle_and_workspace_form(H, Hk, D, B, dtype, ps, P):
    from paged_kv_decode_22_gb300 import ops
    lens = _lens(Hk, ps, P)
    c = _case(31 + P, H, Hk, D, B, lens, dtype)
    ps_got, npart, path, ws = _plan(c, ps)
    assert ps_got == ps and npart == P
    if P == 16 and path != ops.PATH_TC_CLUSTER:
        pytest.skip(f"the device holds fewer than {len(lens) * Hk} clusters of 16 CTAs")
    assert path == ops.PATH_TC_CLUSTER and ws == 0, (npart, path, ws)
    dc = DeviceCase(c)
    got, status = run_decode(dc, partition_size=ps)
    assert status == 0
    ref = _oracle(c)
    assert_close(got, ref, f"cluster H{H}/{Hk} B{B} ps{ps} P{npart}")
    for s, L in enumerate(lens):
        if L == 0:
            assert (got[s] == 0).all()
    # The same partitions merged through the workspace and the merge launch.
    big = 17 * ps
    _, npart2, path2, ws2 = _plan(c, ps, big)
    assert npart2 == 17 and path2 == ops.PATH_TC and ws2 > 0
    got2, status2 = run_decode(dc, partition_size=ps, max_context_len=big)
    assert status2 == 0
    assert_close(got2, ref, "workspace form")
    assert np.abs(got - got2).max() <= 2e-2


def test_library_picks_the_cluster_form_at_batch_one():
    from paged_kv_decode_22_gb300 import ops
    for ctx in (512, 1024, 2048):
        ps, npart, path, ws = ops.decode_plan(1, 64, 8, 128, 16, ctx, 0)
        assert npart > 1 and path == ops.PATH_TC_CLUSTER and ws == 0, (ctx, ps, npart, path)


def test_cluster_bad_block_and_bad_length_set_status_and_zero_rows():
    from paged_kv_decode_22_gb300 import ops
    c = _case(41, 32, 4, 128, 16, [600, 600], "bf16")
    dc = DeviceCase(c)
    assert _plan(c, 128)[2] == ops.PATH_TC_CLUSTER
    bt = c.block_tables.copy()
    bt[1, 20] = c.num_blocks + 9        # a bad id in the second sequence's 3rd partition
    got, status = run_decode(dc, partition_size=128, block_tables=up(bt))
    assert status & 1
    assert (got[1] == 0).all()
    ref = _oracle(c)
    assert_close(got[0], ref[0], "good sequence beside a bad one")

    lens = c.context_lens.copy()
    lens[0] = 601                       # above max_context_len below
    got, status = run_decode(dc, partition_size=128, context_lens=up(lens), max_context_len=600)
    assert status & 4
    assert (got[0] == 0).all()
    assert_close(got[1], ref[1], "good sequence beside a bad length")


def test_cluster_form_with_alibi():
    from paged_kv_decode_22_gb300 import ops
    H, Hk = 48, 1
    lens = [1000, 3, 129, 0, 640]
    c = _case(43, H, Hk, 128, 16, lens, "fp16")
    assert _plan(c, 128)[2] == ops.PATH_TC_CLUSTER
    dc = DeviceCase(c)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32)
    out = torch.full(c.q.shape, float("nan"), dtype=dc.q.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, c.max_context_len, c.scale,
                               partition_size=128, device_status=status,
                               alibi_slopes=torch.from_numpy(slopes).cuda())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = decode_bits(down_bits(out), "fp16")
    assert_close(got, _oracle(c, alibi_slopes=slopes.astype(np.float64)), "alibi, cluster form")


def test_cluster_form_is_repeatable_and_needs_no_workspace():
    from paged_kv_decode_22_gb300 import ops
    c = _case(47, 64, 8, 128, 16, [2048], "bf16")
    dc = DeviceCase(c)
    ps, npart, path, ws = _plan(c, 0)
    assert path == ops.PATH_TC_CLUSTER and ws == 0
    outs = []
    for _ in range(3):
        out = torch.full(c.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, 2048, c.scale,
                                   workspace=None)
        outs.append(out)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert_close(decode_bits(down_bits(outs[0]), "bf16"), _oracle(c), "b1 ctx2048")
