"""Prefill over the paged cache on the GPU (through the C ABI) against the
float64 prefill oracle, outputs decoded from fp16/bf16.

Two kernels serve prefill: the single form (one query tile per work unit)
and the paired form (two query tiles of one sequence and KV head share every
K/V tile), taken when the host's bounds promise long units.  Passing a large
max_context_len (a valid upper bound) selects the paired form, so the tests
run both on the same data.

Tolerance: |err| <= 1e-2 + one ulp of the output type at |ref| (2^-7 |ref|
for bf16, 2^-10 |ref| for fp16) per element, mean |err| <= 1e-3.  The ulp
term is the final rounding itself: the first queries of a chunk without
prefix see a handful of tokens, so |out| reaches |v| (about 4 here), where
rounding the exact result to bf16 already moves it by up to 0.0078.
"""
import numpy as np
import pytest
import torch

from oracle.formats import decode_bits
from oracle.prefill import paged_prefill_attention as oracle_prefill
from paged_kv_decode_22_gb300.workloads import make_prefill_case

from .gpu_util import TORCH_DT, assert_close_ulp, down_bits, up

pytestmark = pytest.mark.gpu

# (H, Hk, B, dtype): query-group sizes 1..64 -> 64/g queries per work unit
LAYOUTS = [(64, 8, 16, "bf16"), (32, 32, 16, "fp16"), (48, 1, 16, "fp16"), (64, 1, 32, "bf16"),
           (16, 4, 64, "bf16"), (40, 8, 16, "fp16"), (24, 8, 256, "fp16"), (32, 16, 8, "bf16")]

# (context length, chunk length): no prefix, prefixed, decode-like, empty,
# chunk ending mid-block, long chunk over a long prefix
CHUNKS = [(300, 300), (1000, 37), (129, 1), (64, 0), (17, 17), (700, 200)]


def _case(seed, H, Hk, B, dtype, chunks, **kw):
    lens = [L for L, _ in chunks]
    need = sum(-(-L // B) for L in lens)
    return make_prefill_case(seed=seed, num_seqs=len(chunks), num_heads=H, num_kv_heads=Hk,
                             head_size=128, block_size=B, num_blocks=need + 6, context_lens=lens,
                             query_lens=[n for _, n in chunks], dtype=dtype, **kw)


# max_context_len that makes the host pick each form for the test chunks
# (the paired form from max_context_len - max_query_len / 2 >= 1024).
FORM_CTX = {"single": None, "pair": 8192}


def _run(c, *, max_query_len=None, max_context_len=None, block_tables=None, context_lens=None,
         alibi=None, form="single", scale=None):
    if max_context_len is None:
        max_context_len = FORM_CTX[form]
    from paged_kv_decode_22_gb300 import ops
    b = c.base
    out = torch.full(c.q.shape, float("nan"), dtype=TORCH_DT[b.dtype], device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.paged_prefill_attention(
        out, up(c.q, b.dtype), up(b.key_cache, b.dtype), up(b.value_cache, b.dtype),
        up(b.block_tables if block_tables is None else block_tables),
        up(b.context_lens if context_lens is None else context_lens), up(c.query_start),
        int(c.query_lens.max()) if max_query_len is None else max_query_len,
        b.max_context_len if max_context_len is None else max_context_len,
        b.scale if scale is None else scale, device_status=status,
        alibi_slopes=None if alibi is None else torch.from_numpy(alibi).cuda())
    torch.cuda.synchronize()
    return decode_bits(down_bits(out), b.dtype), int(status.item())


def _oracle(c, scale=None, **kw):
    b = c.base
    return oracle_prefill(c.q, b.key_cache, b.value_cache, b.block_tables, b.context_lens,
                          c.query_start, b.scale if scale is None else scale, b.dtype, **kw)


@pytest.mark.parametrize("form", ["single", "pair"])
@pytest.mark.parametrize("H,Hk,B,dtype", LAYOUTS)
def test_prefill_matches_oracle(H, Hk, B, dtype, form):
    c = _case(61, H, Hk, B, dtype, CHUNKS)
    got, status = _run(c, form=form)
    assert status == 0
    assert_close_ulp(got, _oracle(c), dtype, f"prefill H{H}/{Hk} B{B} {dtype} {form}")


@pytest.mark.parametrize("H,Hk,B,dtype", [(64, 8, 16, "bf16"), (32, 32, 16, "fp16"),
                                          (64, 1, 32, "bf16"), (24, 8, 256, "fp16")])
def test_paired_form_on_long_prefixes_with_its_own_bounds(H, Hk, B, dtype):
    # Chunks over cached prefixes long enough that the host's own bounds pick
    # the paired form; odd query-tile counts leave a unit with one slot.
    chunks = [(4000, 300), (2500, 77), (1500, 1), (3100, 129), (2048, 0)]
    c = _case(63, H, Hk, B, dtype, chunks)
    assert c.base.max_context_len - 300 // 2 >= 1024
    got, status = _run(c)
    assert status == 0
    assert_close_ulp(got, _oracle(c), dtype, f"paired, long prefixes H{H}/{Hk} B{B}")


def test_both_forms_agree():
    c = _case(65, 64, 8, 16, "bf16", CHUNKS)
    a, _ = _run(c, form="single")
    b, _ = _run(c, form="pair")
    assert np.abs(a - b).max() <= 2e-2


@pytest.mark.parametrize("form", ["single", "pair"])
@pytest.mark.parametrize("H,Hk,B,dtype", [(64, 8, 16, "bf16"), (32, 32, 16, "fp16"),
                                          (48, 1, 16, "fp16")])
def test_prefill_with_alibi(H, Hk, B, dtype, form):
    c = _case(67, H, Hk, B, dtype, [(400, 150), (90, 90), (33, 1)])
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32)
    got, status = _run(c, alibi=slopes, form=form)
    assert status == 0
    assert_close_ulp(got, _oracle(c, alibi_slopes=slopes.astype(np.float64)), dtype,
                     "prefill alibi")


@pytest.mark.parametrize("form", ["single", "pair"])
@pytest.mark.parametrize("scale", [0.0, -0.06])
def test_prefill_with_a_scale_of_zero_or_below(scale, form):
    # Such a scale cannot fold into the exponent (the maximum of the scaled
    # logits is then not the scaled maximum), so these calls run in the
    # kernel instantiation that scales every logit first, the one ALiBi uses.
    c = _case(71, 64, 8, 16, "bf16", [(400, 150), (1500, 256), (33, 1)])
    got, status = _run(c, form=form, scale=scale)
    assert status == 0
    assert_close_ulp(got, _oracle(c, scale=scale), "bf16", f"prefill scale {scale}")


def test_one_query_per_sequence_equals_decode():
    from paged_kv_decode_22_gb300 import ops

    from .gpu_util import DeviceCase
    c = _case(71, 64, 8, 16, "bf16", [(1000, 1), (37, 1), (512, 1), (129, 1)])
    got, status = _run(c)
    assert status == 0
    b = c.base
    b.q = c.q.copy()
    dc = DeviceCase(b)
    out = torch.empty(c.q.shape, dtype=torch.bfloat16, device="cuda")
    ops.paged_decode_attention(out, dc.q, dc.kc, dc.vc, dc.bt, dc.cl, b.max_context_len, b.scale)
    torch.cuda.synchronize()
    dec = decode_bits(down_bits(out), "bf16")
    assert np.abs(got - dec).max() <= 1e-2
    assert_close_ulp(got, _oracle(c), "bf16", "one query per sequence")


@pytest.mark.parametrize("form", ["single", "pair"])
def test_bad_block_zeroes_only_the_queries_that_reach_it(form):
    c = _case(73, 32, 4, 16, "bf16", [(400, 100), (200, 50)])
    good = _oracle(c)
    bt = c.base.block_tables.copy()
    bt[0, 20] = c.base.num_blocks + 5          # tokens 320..335: queries at positions >= 320
    got, status = _run(c, block_tables=bt, form=form)
    assert status & 1
    c.base.block_tables = bt
    ref = _oracle(c)
    assert (ref[:20] == good[:20]).all() and (ref[20:100] == 0).all()
    assert_close_ulp(got, ref, "bf16", "bad block")


def test_invalid_chunks_give_zero_rows_and_set_the_length_bit():
    c = _case(79, 16, 2, 16, "fp16", [(100, 40), (50, 10), (80, 30)])
    lens = c.base.context_lens.copy()
    lens[1] = 5                                  # chunk of 10 longer than the context
    got, status = _run(c, context_lens=lens)
    assert status & 4
    assert (got[40:50] == 0).all()
    c.base.context_lens = lens
    assert_close_ulp(got, _oracle(c), "fp16", "chunk longer than its context")
    c.base.context_lens[1] = 50
    got, status = _run(c, max_query_len=35)      # the 40-token chunk is too long
    assert status & 4
    assert (got[:40] == 0).all()
    assert_close_ulp(got, _oracle(c, max_query_len=35), "fp16", "chunk longer than max_query_len")


@pytest.mark.parametrize("form", ["single", "pair"])
def test_many_sequences_with_multi_tile_chunks_read_the_tables_from_global_memory(form):
    # More than 128 sequences (lengths and chunk bounds read from global
    # memory, not the shared-memory table) with chunks of up to 3 query tiles
    # (g = 8: 16 queries per tile).
    rng = np.random.default_rng(9)
    lens = rng.integers(1, 90, 1100)
    qlens = np.minimum(rng.integers(0, 48, 1100), lens)
    c = _case(87, 16, 2, 16, "bf16", [(int(L), int(n)) for L, n in zip(lens, qlens)])
    got, status = _run(c, form=form)
    assert status == 0
    rows = [(int(r), int(h)) for r, h in zip(np.random.default_rng(10).integers(0, c.q.shape[0], 64),
                                             np.random.default_rng(11).integers(0, 16, 64))]
    ref = _oracle(c, rows=rows)
    assert_close_ulp(np.stack([got[r, h] for r, h in rows]), ref, "bf16", "1100 sequences, multi-tile chunks")


def test_many_sequences_use_the_round_robin_schedule():
    # More than 1024 sequences: units are taken round-robin, not from the
    # shared-memory schedule.
    chunks = [(int(L), int(n)) for L, n in zip(np.random.default_rng(5).integers(1, 40, 1100),
                                               np.random.default_rng(6).integers(0, 5, 1100))]
    chunks = [(L, min(n, L)) for L, n in chunks]
    c = _case(83, 16, 2, 16, "bf16", chunks)
    got, status = _run(c)
    assert status == 0
    rows = [(int(r), int(h)) for r, h in zip(np.random.default_rng(7).integers(0, c.q.shape[0], 64),
                                             np.random.default_rng(8).integers(0, 16, 64))]
    ref = _oracle(c, rows=rows)
    assert_close_ulp(np.stack([got[r, h] for r, h in rows]), ref, "bf16", "1100 sequences")
