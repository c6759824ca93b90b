"""Pins of the prefill oracle (oracle/prefill.py) against things other than itself.

* brute force: pure-Python triple-loop attention of each query over the
  cache rows up to its own position, walked with plain loops;
* closed forms: a zero query averages the visible value rows, so the causal
  window of every query is checked by its mean; the first query of a chunk
  without prefix returns its own value row exactly;
* reductions: one query per sequence is decode; the last query of a chunk is
  decode over the whole context;
* invariants: changing cache rows after a query's position leaves its output
  alone and changes the queries that see them; invalid chunks give zeros;
* planted mistakes in the position and window helpers are caught.
"""
import numpy as np
import pytest

import oracle.prefill as pf
from oracle.brute import dense_decode_attention
from oracle.formats import decode_bits
from oracle.paged_attention import paged_decode_attention
from oracle.prefill import paged_prefill_attention
from paged_kv_decode_22_gb300.workloads import f32_to_bf16_bits, make_prefill_case


def _run(c, **kw):
    b = c.base
    return paged_prefill_attention(c.q, b.key_cache, b.value_cache, b.block_tables,
                                   b.context_lens, c.query_start, b.scale, b.dtype, **kw)


def _rows(cache, table, L, B, kv, dtype):
    out = []
    for t in range(L):
        blk = int(table[t // B])
        out.append([float(v) for v in decode_bits(cache[blk, t - (t // B) * B, kv], dtype)])
    return out


@pytest.mark.parametrize("seed,H,Hk,D,B,lens,qlens,dtype,alibi", [
    (1, 4, 2, 8, 4, [7, 13, 5], [3, 13, 1], "fp16", False),
    (2, 6, 1, 16, 8, [20, 9], [5, 9], "bf16", False),
    (3, 4, 4, 12, 4, [11, 6], [4, 2], "bf16", True),
    (4, 8, 2, 16, 16, [33, 17, 2], [16, 1, 2], "fp16", True),
])
def test_prefill_oracle_matches_brute_force(seed, H, Hk, D, B, lens, qlens, dtype, alibi):
    c = make_prefill_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                          head_size=D, block_size=B, num_blocks=24, context_lens=lens,
                          query_lens=qlens, dtype=dtype)
    slopes = [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)] if alibi else None
    out = _run(c, alibi_slopes=slopes)
    b = c.base
    g = H // Hk
    for s, (L, n) in enumerate(zip(lens, qlens)):
        for i in range(n):
            r = int(c.query_start[s]) + i
            p = L - n + i
            for h in range(H):
                K = _rows(b.key_cache, b.block_tables[s], p + 1, B, h // g, dtype)
                V = _rows(b.value_cache, b.block_tables[s], p + 1, B, h // g, dtype)
                qv = [float(v) for v in decode_bits(c.q[r, h], dtype)]
                ref = dense_decode_attention(qv, K, V, b.scale, slopes[h] if alibi else 0.0)
                np.testing.assert_allclose(out[r, h], ref, rtol=0, atol=1e-12)
    assert np.isfinite(out).all()


def test_zero_query_averages_exactly_the_visible_rows():
    lens, qlens = [9, 6, 12], [4, 6, 1]
    c = make_prefill_case(seed=5, num_seqs=3, num_heads=2, num_kv_heads=1, head_size=8,
                          block_size=4, num_blocks=16, context_lens=lens, query_lens=qlens,
                          dtype="bf16")
    c.q[:] = f32_to_bf16_bits(np.zeros(1, np.float32))[0]
    out = _run(c)
    b = c.base
    for s, (L, n) in enumerate(zip(lens, qlens)):
        V = np.array(_rows(b.value_cache, b.block_tables[s], L, 4, 0, "bf16"))
        for i in range(n):
            r = int(c.query_start[s]) + i
            want = V[:L - n + i + 1].mean(axis=0)
            for h in range(2):
                np.testing.assert_allclose(out[r, h], want, rtol=0, atol=1e-12)


def test_first_query_without_prefix_returns_its_value_row():
    c = make_prefill_case(seed=6, num_seqs=2, num_heads=4, num_kv_heads=2, head_size=16,
                          block_size=8, num_blocks=8, context_lens=[10, 3], query_lens=[10, 3],
                          dtype="fp16")
    out = _run(c)
    b = c.base
    for s in range(2):
        r = int(c.query_start[s])
        for h in range(4):
            v0 = decode_bits(b.value_cache[b.block_tables[s, 0], 0, h // 2], "fp16")
            np.testing.assert_array_equal(out[r, h], v0)


def test_one_query_per_sequence_is_decode():
    c = make_prefill_case(seed=7, num_seqs=4, num_heads=8, num_kv_heads=2, head_size=16,
                          block_size=4, num_blocks=32, context_lens=[1, 5, 19, 0],
                          query_lens=[1, 1, 1, 0], dtype="bf16")
    b = c.base
    out = _run(c)
    q_dec = b.q.copy()
    q_dec[:3] = c.q
    ref = paged_decode_attention(q_dec, b.key_cache, b.value_cache, b.block_tables,
                                 b.context_lens, b.scale, "bf16")
    np.testing.assert_array_equal(out, ref[:3])


def test_last_query_of_a_chunk_is_decode_over_the_whole_context():
    c = make_prefill_case(seed=8, num_seqs=2, num_heads=4, num_kv_heads=1, head_size=16,
                          block_size=8, num_blocks=16, context_lens=[30, 17],
                          query_lens=[7, 17], dtype="fp16")
    b = c.base
    out = _run(c)
    last = c.query_start[1:] - 1
    q_dec = c.q[last]
    ref = paged_decode_attention(q_dec, b.key_cache, b.value_cache, b.block_tables,
                                 b.context_lens, b.scale, "fp16")
    np.testing.assert_array_equal(out[last], ref)


def test_later_cache_rows_do_not_reach_earlier_queries():
    c = make_prefill_case(seed=9, num_seqs=1, num_heads=2, num_kv_heads=1, head_size=8,
                          block_size=4, num_blocks=8, context_lens=[14], query_lens=[6],
                          dtype="fp16")
    b = c.base
    before = _run(c)
    t = 11                                   # position of query 3 (14 - 6 + 3)
    blk = b.block_tables[0, t // 4]
    b.key_cache[blk, t % 4] ^= np.uint16(0x1234)
    b.value_cache[blk, t % 4] ^= np.uint16(0x0F0F)
    after = _run(c)
    np.testing.assert_array_equal(after[:3], before[:3])
    assert np.all(np.abs(after[3:] - before[3:]).max(axis=(1, 2)) > 0)


def test_invalid_chunks_give_zero_rows_and_empty_chunks_give_none():
    c = make_prefill_case(seed=10, num_seqs=3, num_heads=2, num_kv_heads=2, head_size=8,
                          block_size=4, num_blocks=16, context_lens=[5, 8, 3],
                          query_lens=[2, 0, 3], dtype="bf16")
    b = c.base
    b.context_lens[0] = 1                   # chunk of 2 longer than the context
    out = _run(c)
    assert out.shape == (5, 2, 8)
    assert (out[:2] == 0).all()
    assert np.isfinite(out[2:]).all() and np.abs(out[2:]).max() > 0
    b.block_tables[2, 0] = 99               # a bad block id under every query
    out = _run(c)
    assert (out[2:] == 0).all()


def test_chunks_longer_than_max_query_len_give_zero_rows_and_others_are_unchanged():
    # Reading of the invalid-input rule: a chunk longer than the caller's
    # max_query_len is invalid (all its rows zero); a chunk of exactly
    # max_query_len is attended, and no other sequence is affected.
    c = make_prefill_case(seed=13, num_seqs=3, num_heads=4, num_kv_heads=2, head_size=8,
                          block_size=4, num_blocks=24, context_lens=[9, 6, 12],
                          query_lens=[4, 5, 3], dtype="fp16")
    full = _run(c)
    out = _run(c, max_query_len=4)
    assert np.abs(full[4:9]).max() > 0                     # the 5-query chunk, unlimited
    assert (out[4:9] == 0).all()                           # ... and over the limit
    np.testing.assert_array_equal(out[:4], full[:4])       # n == max_query_len: attended
    np.testing.assert_array_equal(out[9:], full[9:])
    out = _run(c, max_query_len=5)
    np.testing.assert_array_equal(out, full)


def test_a_bad_block_zeroes_only_the_queries_that_see_it():
    c = make_prefill_case(seed=12, num_seqs=1, num_heads=2, num_kv_heads=1, head_size=8,
                          block_size=4, num_blocks=16, context_lens=[20], query_lens=[10],
                          dtype="fp16")
    b = c.base
    good = _run(c)
    b.block_tables[0, 3] = -7               # tokens 12..15: queries at positions >= 12
    out = _run(c)
    np.testing.assert_array_equal(out[:2], good[:2])      # positions 10, 11
    assert (out[2:] == 0).all()                            # positions 12..19


def test_sampled_rows_equal_full_output():
    c = make_prefill_case(seed=11, num_seqs=2, num_heads=4, num_kv_heads=2, head_size=8,
                          block_size=4, num_blocks=16, context_lens=[10, 7],
                          query_lens=[4, 3], dtype="fp16")
    full = _run(c)
    rows = [(6, 3), (0, 0), (3, 1), (4, 2)]
    got = _run(c, rows=rows)
    for k, (r, h) in enumerate(rows):
        np.testing.assert_allclose(got[k], full[r, h], rtol=0, atol=1e-14)


def _pins():
    test_prefill_oracle_matches_brute_force(1, 4, 2, 8, 4, [7, 13, 5], [3, 13, 1], "fp16", False)
    test_zero_query_averages_exactly_the_visible_rows()
    test_first_query_without_prefix_returns_its_value_row()
    test_later_cache_rows_do_not_reach_earlier_queries()


@pytest.mark.parametrize("attr,fn", [
    ("query_position", lambda L, n, i: L - n + i + 1),      # one past its own position
    ("query_position", lambda L, n, i: L - n + i - 1),      # one short
    ("query_position", lambda L, n, i: i),                  # measured from the chunk start
    ("query_position", lambda L, n, i: L - 1),              # every query at the end
    ("visible_tokens", lambda p: p),                        # excludes itself
    ("visible_tokens", lambda p: p + 2),                    # sees the next token
], ids=["pos+1", "pos-1", "pos_from_chunk", "pos_at_end", "exclusive", "one_ahead"])
def test_pins_catch_planted_prefill_mistakes(attr, fn, monkeypatch):
    monkeypatch.setattr(pf, attr, fn)
    with pytest.raises((AssertionError, IndexError, ValueError, FloatingPointError)):
        with np.errstate(all="raise"):
            _pins()
