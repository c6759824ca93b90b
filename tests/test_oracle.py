"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-evaluated golden case (tests/golden/hand_paged_gqa.json);
* exact format constants for fp16 / bf16 decoding;
* a pure-Python brute-force dense attention on contiguous K/V, with the
  contiguous rows collected by walking the block table in plain loops;
* closed forms: one token returns its V, identical keys or scale 0 return the
  mean of V, a dominant logit returns that token's V;
* invariants: permuting physical blocks (with a matching table), GQA equal to
  MHA with repeated KV heads, V shifted by a constant, split-context merge
  equal to the unsplit softmax;
* gather / cache: a pool whose rows encode their own slot number.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle.brute import dense_decode_attention
from oracle.cache import cache_kv
from oracle.formats import decode_bits
from oracle.gather import gather_cached_kv
from oracle.paged_attention import kv_head_of, paged_decode_attention
from oracle.split_context import merge, partial, split_attention
from paged_kv_decode_22_gb300.workloads import (
    f32_to_bf16_bits, f32_to_f16_bits, make_decode_case, make_gather_case)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x, dtype):
    return f32_to_f16_bits(np.asarray(x, np.float32)) if dtype == "fp16" else \
        f32_to_bf16_bits(np.asarray(x, np.float32))


def _load_hand_case():
    with open(os.path.join(GOLDEN, "hand_paged_gqa.json")) as f:
        g = json.load(f)
    nan = float("nan")

    def arr(v):
        def fill(x):
            if x is None:
                return [nan] * g["head_size"]
            if isinstance(x, list):
                return [fill(y) for y in x]
            return x
        return np.array(fill(v), dtype=np.float32)

    return g, _bits(arr(g["q"]), "fp16"), _bits(arr(g["key_cache"]), "fp16"), \
        _bits(arr(g["value_cache"]), "fp16")


# ---------------------------------------------------------------- formats

@pytest.mark.parametrize("bits,val", [(0x3C00, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -24),
                                      (0x7BFF, 65504.0), (0x3555, 0.333251953125)])
def test_fp16_decode_constants(bits, val):
    assert decode_bits(np.array([bits], np.uint16), "fp16")[0] == val


@pytest.mark.parametrize("bits,val", [(0x3F80, 1.0), (0xC040, -3.0), (0x0001, 2.0 ** -133),
                                      (0x3EAB, 0.333984375), (0x7F7F, 3.3895313892515355e38)])
def test_bf16_decode_constants(bits, val):
    assert decode_bits(np.array([bits], np.uint16), "bf16")[0] == val


def test_bf16_encoder_rounds_to_nearest_even():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6... and goes to 1 + 2^-6 (even).
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -2.5], np.float32)
    got = decode_bits(f32_to_bf16_bits(x), "bf16")
    assert got.tolist() == [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -2.5]


# ---------------------------------------------------------------- golden

def test_hand_case_golden():
    g, q, kc, vc = _load_hand_case()
    out = paged_decode_attention(q, kc, vc, np.array(g["block_tables"], np.int32),
                                 np.array(g["context_lens"], np.int32), math.log(2.0), "fp16")
    np.testing.assert_allclose(out, np.array(g["expected_out"], np.float64), rtol=0, atol=1e-14)


def test_hand_case_kv_head_mapping_is_contiguous():
    assert [kv_head_of(h, 4, 2) for h in range(4)] == [0, 0, 1, 1]
    assert [kv_head_of(h, 48, 1) for h in (0, 17, 47)] == [0, 0, 0]
    assert [kv_head_of(h, 64, 8) for h in (0, 7, 8, 63)] == [0, 0, 1, 7]


def test_hand_alibi_golden():
    with open(os.path.join(GOLDEN, "hand_alibi.json")) as f:
        g = json.load(f)
    nan = float("nan")

    def arr(v):
        def fill(x):
            if x is None:
                return nan
            if isinstance(x, list):
                return [fill(y) for y in x]
            return x
        return np.array(fill(v), dtype=np.float32)

    slopes = [math.log(2.0) if v == "ln2" else v for v in g["alibi_slopes"]]
    out = paged_decode_attention(_bits(arr(g["q"]), "fp16"), _bits(arr(g["key_cache"]), "fp16"),
                                 _bits(arr(g["value_cache"]), "fp16"),
                                 np.array(g["block_tables"], np.int32),
                                 np.array(g["context_lens"], np.int32), g["scale"], "fp16",
                                 alibi_slopes=slopes)
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-14)


def test_alibi_with_zero_slopes_is_plain_attention():
    c = _case(lens=(6, 21), H=6, Hk=2, D=8)
    base = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                  c.context_lens, c.scale, "fp16")
    zero = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                  c.context_lens, c.scale, "fp16", alibi_slopes=np.zeros(6))
    np.testing.assert_array_equal(base, zero)


# ---------------------------------------------------------------- brute force

def _contiguous_rows(cache, table, L, B, kv, dtype):
    """Walk the block table with plain loops (independent of the oracle's indexing)."""
    rows = []
    for t in range(L):
        blk = int(table[t // B])
        off = t - (t // B) * B
        rows.append([float(v) for v in decode_bits(cache[blk, off, kv], dtype)])
    return rows


@pytest.mark.parametrize("seed,H,Hk,D,B,lens,dtype", [
    (1, 4, 4, 8, 4, [1, 7, 13], "fp16"),
    (2, 6, 2, 16, 8, [9, 24], "bf16"),
    (3, 8, 1, 12, 16, [40, 17, 33], "fp16"),
    (4, 4, 2, 64, 16, [17, 40], "bf16"),
])
def test_oracle_matches_brute_force(seed, H, Hk, D, B, lens, dtype):
    c = make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                         head_size=D, block_size=B, num_blocks=16, context_lens=lens,
                         dtype=dtype)
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, dtype)
    g = H // Hk
    for s, L in enumerate(lens):
        for h in range(H):
            kv = h // g
            K = _contiguous_rows(c.key_cache, c.block_tables[s], L, B, kv, dtype)
            V = _contiguous_rows(c.value_cache, c.block_tables[s], L, B, kv, dtype)
            qv = [float(v) for v in decode_bits(c.q[s, h], dtype)]
            ref = dense_decode_attention(qv, K, V, c.scale)
            np.testing.assert_allclose(out[s, h], ref, rtol=0, atol=1e-12)
    assert np.isfinite(out).all()  # poisoned (NaN) slots were never read


@pytest.mark.parametrize("seed,H,Hk,lens", [(21, 4, 2, [5, 19]), (22, 8, 1, [33, 1, 12])])
def test_oracle_with_alibi_matches_brute_force(seed, H, Hk, lens):
    c = make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                         head_size=16, block_size=8, num_blocks=16, context_lens=lens,
                         dtype="bf16")
    slopes = [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "bf16", alibi_slopes=slopes)
    g = H // Hk
    for s, L in enumerate(lens):
        for h in range(H):
            K = _contiguous_rows(c.key_cache, c.block_tables[s], L, 8, h // g, "bf16")
            V = _contiguous_rows(c.value_cache, c.block_tables[s], L, 8, h // g, "bf16")
            qv = [float(v) for v in decode_bits(c.q[s, h], "bf16")]
            ref = dense_decode_attention(qv, K, V, c.scale, slopes[h])
            np.testing.assert_allclose(out[s, h], ref, rtol=0, atol=1e-12)


def test_sampled_pairs_equal_full_output():
    c = make_decode_case(seed=7, num_seqs=3, num_heads=8, num_kv_heads=2, head_size=16,
                         block_size=4, num_blocks=32, context_lens=[5, 0, 30], dtype="bf16")
    full = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                  c.context_lens, c.scale, "bf16")
    pairs = [(2, 7), (0, 0), (1, 3), (2, 4)]
    got = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "bf16", pairs=pairs)
    for i, (s, h) in enumerate(pairs):
        np.testing.assert_allclose(got[i], full[s, h], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- closed forms

def _case(seed=11, lens=(1, 5, 19), H=4, Hk=2, D=16, B=4, dtype="fp16", **kw):
    return make_decode_case(seed=seed, num_seqs=len(lens), num_heads=H, num_kv_heads=Hk,
                            head_size=D, block_size=B, num_blocks=24, context_lens=list(lens),
                            dtype=dtype, **kw)


def test_single_token_returns_its_value_row():
    c = _case(lens=(1, 1))
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "fp16")
    for s in range(2):
        for h in range(4):
            v = decode_bits(c.value_cache[c.block_tables[s, 0], 0, h // 2], "fp16")
            np.testing.assert_array_equal(out[s, h], v)


def test_identical_keys_give_mean_of_values():
    c = _case(lens=(7, 13))
    c.key_cache[:] = c.key_cache[c.block_tables[0, 0], 0][None, None]
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "fp16")
    for s, L in enumerate((7, 13)):
        for h in range(4):
            t = np.arange(L)
            V = decode_bits(c.value_cache[c.block_tables[s, t // 4], t % 4, h // 2], "fp16")
            np.testing.assert_allclose(out[s, h], V.mean(axis=0), rtol=0, atol=1e-14)


def test_zero_scale_gives_mean_of_values():
    c = _case(lens=(9,), poison=False)
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, 0.0, "fp16")
    t = np.arange(9)
    for h in range(4):
        V = decode_bits(c.value_cache[c.block_tables[0, t // 4], t % 4, h // 2], "fp16")
        np.testing.assert_allclose(out[0, h], V.mean(axis=0), rtol=0, atol=1e-14)


def test_dominant_logit_returns_that_value_row():
    # q = K[t*] scaled up: logit gap >= 700 nats, so every other weight underflows to 0.
    c = _case(lens=(11,), D=8, poison=False, dtype="bf16")
    t_star = 6
    blk, off = c.block_tables[0, t_star // 4], t_star % 4
    k = decode_bits(c.key_cache[blk, off, 0], "bf16")
    c.key_cache[:, :, 0] = 0
    c.key_cache[blk, off, 0] = f32_to_bf16_bits(np.full(8, 1.0, np.float32))
    c.q[0, 0] = f32_to_bf16_bits(np.full(8, 1.0, np.float32))
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, 100.0, "bf16", pairs=[(0, 0)])
    np.testing.assert_array_equal(out[0], decode_bits(c.value_cache[blk, off, 0], "bf16"))
    assert k.shape == (8,)


def test_zero_length_gives_zeros_and_empty_pairs():
    c = _case(lens=(0, 3))
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "fp16")
    assert (out[0] == 0).all() and np.isfinite(out).all()


# ---------------------------------------------------------------- invariants

def test_block_permutation_invariance():
    c = _case(lens=(5, 19, 12), poison=False)
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "fp16")
    perm = np.random.default_rng(3).permutation(c.num_blocks)
    inv = np.argsort(perm)
    kc2 = c.key_cache[perm]        # physical block j now holds old block perm[j]
    vc2 = c.value_cache[perm]
    bt2 = inv[c.block_tables].astype(np.int32)
    out2 = paged_decode_attention(c.q, kc2, vc2, bt2, c.context_lens, c.scale, "fp16")
    np.testing.assert_array_equal(out, out2)


def test_gqa_equals_mha_with_repeated_kv_heads():
    c = _case(lens=(6, 21), H=6, Hk=2, D=8)
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "fp16")
    kc = np.repeat(c.key_cache, 3, axis=2)
    vc = np.repeat(c.value_cache, 3, axis=2)
    out_mha = paged_decode_attention(c.q, kc, vc, c.block_tables, c.context_lens, c.scale,
                                     "fp16")
    np.testing.assert_allclose(out, out_mha, rtol=0, atol=1e-15)


def test_value_shift_shifts_output():
    c = _case(lens=(13,), poison=False, dtype="bf16")
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "bf16")
    shift = 3.0  # adding 3 to a bf16 of magnitude < 8 ... compare in float64 after decoding
    vals = decode_bits(c.value_cache, "bf16") + shift
    vc2 = f32_to_bf16_bits(vals.astype(np.float32))
    base = paged_decode_attention(c.q, c.key_cache, vc2, c.block_tables, c.context_lens,
                                  c.scale, "bf16")
    # vc2 is vals rounded; compare against the softmax-weighted rounding error bound.
    err = np.abs(decode_bits(vc2, "bf16") - vals).max()
    assert np.abs(base - (out + shift)).max() <= err + 1e-12


def test_split_context_merge_equals_unsplit():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(200) * 3
    V = rng.standard_normal((200, 16))
    w = np.exp(x - x.max())
    ref = (w @ V) / w.sum()
    for bounds in ([0, 200], [0, 1, 200], [0, 64, 128, 192, 200], [0, 50, 50, 199, 200]):
        np.testing.assert_allclose(split_attention(x, V, bounds), ref, rtol=0, atol=1e-13)
    o, m, l = partial(x, V)
    assert m == x.max()
    np.testing.assert_allclose(merge([(o, m, l)]), ref, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- gather / cache

def _coded_pool(NB, B, H, D):
    """Pool whose every element holds its own slot number (fits in 16 bits)."""
    slot = np.arange(NB * B, dtype=np.uint16).reshape(NB, B, 1, 1)
    return np.broadcast_to(slot, (NB, B, H, D)).copy(), \
        np.broadcast_to(slot ^ np.uint16(0x8000), (NB, B, H, D)).copy()


def test_gather_returns_the_rows_of_the_listed_slots():
    kc, vc = _coded_pool(64, 8, 3, 4)
    slots = np.array([0, 7, 8, 511, 100, 263], np.int64)
    k, v = gather_cached_kv(kc, vc, slots)
    assert (k == slots.astype(np.uint16)[:, None, None]).all()
    assert (v == (slots.astype(np.uint16) ^ 0x8000)[:, None, None]).all()


def test_gather_invalid_slots_give_zero_rows():
    kc, vc = _coded_pool(4, 8, 2, 2)
    k, v = gather_cached_kv(kc, vc, np.array([-1, 32, 5], np.int64))
    assert (k[:2] == 0).all() and (v[:2] == 0).all() and (k[2] == 5).all()


def test_gather_then_dense_attention_equals_paged_attention():
    # Links the two operations: gathering a sequence's slots gives the K/V rows
    # that paged attention reads.
    c = _case(lens=(19,), poison=False)
    t = np.arange(19)
    slots = c.block_tables[0, t // 4].astype(np.int64) * 4 + t % 4
    k, v = gather_cached_kv(c.key_cache, c.value_cache, slots)
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                 c.context_lens, c.scale, "fp16")
    for h in range(4):
        K = [[float(a) for a in decode_bits(k[i, h // 2], "fp16")] for i in range(19)]
        V = [[float(a) for a in decode_bits(v[i, h // 2], "fp16")] for i in range(19)]
        qv = [float(a) for a in decode_bits(c.q[0, h], "fp16")]
        np.testing.assert_allclose(out[0, h], dense_decode_attention(qv, K, V, c.scale),
                                   rtol=0, atol=1e-12)


def test_cache_then_gather_round_trip():
    g = make_gather_case(seed=9, num_tokens=40, num_heads=2, head_size=8, block_size=8,
                         num_blocks=16, dtype="fp16")
    rng = np.random.default_rng(1)
    key = rng.integers(0, 2 ** 16, (40, 2, 8), dtype=np.uint16)
    val = rng.integers(0, 2 ** 16, (40, 2, 8), dtype=np.uint16)
    kc, vc = cache_kv(key, val, g.key_cache, g.value_cache, g.slot_mapping)
    k2, v2 = gather_cached_kv(kc, vc, g.slot_mapping)
    np.testing.assert_array_equal(k2, key)
    np.testing.assert_array_equal(v2, val)
    untouched = np.ones(16 * 8, bool)
    untouched[g.slot_mapping] = False
    np.testing.assert_array_equal(kc.reshape(128, 2, 8)[untouched],
                                  g.key_cache.reshape(128, 2, 8)[untouched])


def test_cache_skips_negative_and_out_of_range_slots():
    kc, vc = _coded_pool(2, 4, 1, 2)
    key = np.full((3, 1, 2), 0xABCD, np.uint16)
    kc2, vc2 = cache_kv(key, key, kc, vc, np.array([-1, 8, 3], np.int64))
    assert (kc2[0, 3] == 0xABCD).all()
    kc2[0, 3] = kc[0, 3]
    np.testing.assert_array_equal(kc2, kc)


# ---------------------------------------------------------------- invalid sequences

def test_invalid_sequences_give_zero_rows():
    c = _case(lens=(5, 7, 9), poison=False)
    bt = c.block_tables.copy()
    bt[1, 1] = c.num_blocks            # out-of-range block id referenced by seq 1
    lens = c.context_lens.copy()
    lens[2] = bt.shape[1] * 4 + 1      # longer than the table
    out = paged_decode_attention(c.q, c.key_cache, c.value_cache, bt, lens, c.scale, "fp16")
    assert (out[1] == 0).all() and (out[2] == 0).all() and (out[0] != 0).any()
    out2 = paged_decode_attention(c.q, c.key_cache, c.value_cache, c.block_tables,
                                  c.context_lens, c.scale, "fp16", max_context_len=8)
    assert (out2[2] == 0).all() and (out2[0] != 0).any()
