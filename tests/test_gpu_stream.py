"""Stream form of the tensor-core decode (PKD_PATH_TC_STREAM).

One CTA per SM takes an equal contiguous share of the (sequence, KV head)
major list of 128-token tiles; a (sequence, KV head) whose tiles straddle a
share's edge leaves partials in per-CTA slots that a second launch merges
with the log-sum-exp rule of the split-context form ("Paged attention V2"
in "[Performance] Support MQA/GQA in decode phase by using FlashAttention",
vLLM pull request 2744).  Each case forces the form (partition_size = -1),
checks through decode_plan that it is the one that runs, and compares with
the float64 oracle (max |err| <= 1e-2, mean <= 1e-3) and with the
fixed-partition form of the same call.  Length mixes cover fewer tiles than
CTAs (most shares empty or one tile), a few tiles per CTA (pairs cut at both
ends and pairs spanning many shares) and many short sequences.
"""
import numpy as np
import pytest
import torch

from oracle.formats import decode_bits
from oracle.paged_attention import paged_decode_attention as oracle_attention
from paged_kv_decode_22_gb300.workloads import make_decode_case

from .gpu_util import DeviceCase, assert_close, down_bits, run_decode, up

pytestmark = pytest.mark.gpu

STREAM = -1

# (H, Hk, B, dtype): group sizes 4..64 (padded 16/32/48/64), block sizes 16..256
LAYOUTS = [(64, 8, 16, "bf16"), (48, 1, 16, "fp16"), (16, 4, 64, "bf16"), (40, 1, 32, "fp16"),
           (32, 1, 128, "bf16"), (4, 1, 256, "fp16"), (24, 2, 16, "fp16"), (48, 4, 16, "bf16")]


def _lens(kind, Hk):
    if kind == "few_tiles":            # fewer tiles than CTAs
        return [1000, 1, 0, 129, 300]
    if kind == "long":                 # pairs spanning many shares, cut at both ends
        return [8192 // Hk, 6000 // Hk + 3, 100, 7777 // Hk, 0, 129]
    rng = np.random.default_rng(Hk)    # "many": about four tiles per CTA in all
    lens = rng.integers(0, 3200 // Hk + 2, 48)
    lens[:3] = [0, 1, 3200 // Hk]
    return [int(L) for L in lens]


def _case(seed, H, Hk, B, lens, dtype):
    need = sum(-(-L // B) for L in lens)
    return make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                            head_size=128, block_size=B, num_blocks=need + 5, context_lens=lens,
                            dtype=dtype)


def _oracle(c, **kw):
    return oracle_attention(c.q, c.key_cache, c.value_cache, c.block_tables, c.context_lens,
                            c.scale, c.dtype, **kw)


def _plan(c, ps, max_ctx=None):
    from paged_kv_decode_22_gb300 import ops
    return ops.decode_plan(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_size, c.block_size,
                           max_ctx or c.max_context_len, ps)


@pytest.mark.parametrize("H,Hk,B,dtype", LAYOUTS)
@pytest.mark.parametrize("kind", ["few_tiles", "long", "many"])
def test_stream_matches_oracle_and_partition_form(H, Hk, B, dtype, kind):
    from paged_kv_decode_22_gb300 import ops
    lens = _lens(kind, Hk)
    c = _case(101 + Hk, H, Hk, B, lens, dtype)
    ps, npart, path, ws = _plan(c, STREAM)
    assert (ps, npart, path) == (128, 1, ops.PATH_TC_STREAM) and ws > 0
    dc = DeviceCase(c)
    got, status = run_decode(dc, partition_size=STREAM)
    assert status == 0
    ref = _oracle(c)
    assert_close(got, ref, f"stream H{H}/{Hk} B{B} {kind}")
    for s, L in enumerate(lens):
        if L == 0:
            assert (got[s] == 0).all()
    got2, status2 = run_decode(dc, partition_size=128)
    assert status2 == 0
    assert np.abs(got - got2).max() <= 2e-2


def test_stream_at_its_sequence_limit():
    # 1024 sequences (the most the in-kernel prefix holds), lengths 0..300:
    # many pairs per share, every kind of range edge; sampled rows.
    from .gpu_util import sample_pairs
    rng = np.random.default_rng(131)
    lens = [int(L) for L in rng.integers(0, 301, 1024)]
    lens[:3] = [0, 1, 300]
    c = _case(137, 32, 4, 16, lens, "bf16")
    from paged_kv_decode_22_gb300 import ops
    assert _plan(c, STREAM)[2] == ops.PATH_TC_STREAM
    got, status = run_decode(DeviceCase(c), partition_size=STREAM)
    assert status == 0
    pairs = sample_pairs(c, 96, seed=3)
    ref = _oracle(c, pairs=pairs)
    assert_close(np.stack([got[s_, h] for s_, h in pairs]), ref, "1024 sequences, stream form")
    for s_, L in enumerate(lens):
        if L == 0:
            assert (got[s_] == 0).all()


def test_stream_is_repeatable():
    c = _case(107, 64, 8, 16, _lens("many", 8), "bf16")
    dc = DeviceCase(c)
    outs = [run_decode(dc, partition_size=STREAM)[0] for _ in range(3)]
    assert all((outs[0] == o).all() for o in outs[1:])


def test_stream_bad_block_and_bad_length_zero_only_their_sequences():
    c = _case(109, 48, 1, 16, [5000, 4000, 3000], "fp16")
    dc = DeviceCase(c)
    ref = _oracle(c)
    bt = c.block_tables.copy()
    bt[1, 100] = c.num_blocks + 3      # tokens 1600..1615 of the middle sequence
    got, status = run_decode(dc, partition_size=STREAM, block_tables=up(bt))
    assert status & 1
    assert (got[1] == 0).all()
    assert_close(got[[0, 2]], ref[[0, 2]], "sequences beside a bad block")

    lens = c.context_lens.copy()
    lens[0] = 5001                     # above max_context_len below
    got, status = run_decode(dc, partition_size=STREAM, context_lens=up(lens),
                             max_context_len=5000)
    assert status & 4
    assert (got[0] == 0).all()
    assert_close(got[1:], ref[1:], "sequences beside a bad length")


def test_stream_all_empty_gives_zeros():
    c = _case(113, 32, 4, 16, [0, 0, 0], "bf16")
    got, status = run_decode(DeviceCase(c), partition_size=STREAM, max_context_len=64)
    assert status == 0 and (got == 0).all()


def test_stream_with_alibi():
    from paged_kv_decode_22_gb300 import ops
    H, Hk = 48, 1
    lens = [7000, 3, 129, 0, 2640]
    c = _case(127, H, Hk, 16, lens, "fp16")
    dc = DeviceCase(c)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32)
    out = torch.full(c.q.shape, float("nan"), dtype=dc.q.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, c.max_context_len, c.scale,
                               partition_size=STREAM, device_status=status,
                               alibi_slopes=torch.from_numpy(slopes).cuda())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = decode_bits(down_bits(out), "fp16")
    assert_close(got, _oracle(c, alibi_slopes=slopes.astype(np.float64)), "alibi, stream form")


def test_stream_form_is_refused_where_it_cannot_run():
    from paged_kv_decode_22_gb300 import ops
    with pytest.raises(ops.PkdError):    # more sequences than the in-kernel prefix holds
        ops.decode_plan(1025, 32, 4, 128, 16, 512, STREAM)
    with pytest.raises(ops.PkdError):    # query groups below 4 take the CUDA-core path
        ops.decode_plan(8, 32, 32, 128, 16, 512, STREAM)
    with pytest.raises(ops.PkdError):    # head size 64 takes the CUDA-core path
        ops.decode_plan(8, 32, 4, 64, 16, 512, STREAM)
    assert ops.decode_plan(1024, 32, 4, 128, 16, 512, STREAM)[2] == ops.PATH_TC_STREAM
