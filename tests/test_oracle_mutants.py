"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each.

Every mutant below replaces one piece of the oracle; the pins of
test_oracle.py are re-run against it and at least one must fail.  (Moving
the ALiBi origin, e.g. slope * t instead of slope * (t - L + 1), is not a
mistake: it adds a constant per head, which the softmax cancels.)
"""
import math

import numpy as np
import pytest

import oracle.paged_attention as pa
from oracle.formats import decode_bits

from . import test_oracle as pins


def _m_strided_heads(h, H, Hk):
    return h % Hk


def _m_swapped_block_index(cache, table, s, L, kv, dtype):
    B = cache.shape[1]
    t = np.arange(L)
    nb = -(-L // B)
    phys = np.asarray(table[s], np.int64)[np.minimum(t % B, nb - 1)]
    return decode_bits(cache[phys, np.minimum(t // B, B - 1), kv, :], dtype)


def _m_alibi_slope_dropped(slopes, heads, L):
    t = np.arange(L, dtype=np.float64) - (L - 1)
    return np.ones((len(heads), 1)) * t[None, :]


def _m_alibi_wrong_head(slopes, heads, L):
    return pa.__dict__["_orig_alibi"](slopes, [0] * len(heads), L)


def _m_alibi_sign(slopes, heads, L):
    return -pa.__dict__["_orig_alibi"](slopes, heads, L)


def _m_tail_off_by_one(cache, table, s, L, kv, dtype):
    B = cache.shape[1]
    t = np.arange(1, L + 1)
    t = np.minimum(t, -(-L // B) * B - 1)
    phys = np.asarray(table[s], np.int64)[t // B]
    return np.nan_to_num(decode_bits(cache[phys, t % B, kv, :], dtype))


def _m_no_scale(Q, K, V, scale, bias=None):
    X = Q @ K.T
    P = np.exp(X - X.max(axis=1, keepdims=True))
    return (P @ V) / P.sum(axis=1, keepdims=True)


def _m_divide_by_length(Q, K, V, scale, bias=None):
    X = scale * (Q @ K.T)
    P = np.exp(X - X.max(axis=1, keepdims=True))
    return (P @ V) / K.shape[0]


def _m_wrong_sign(Q, K, V, scale, bias=None):
    return pa.__dict__["_orig_attend"](Q, K, V, -scale, bias)


def _m_softmax_over_heads(Q, K, V, scale, bias=None):
    X = scale * (Q @ K.T)
    P = np.exp(X - X.max(axis=0, keepdims=True))
    return (P @ V) / P.sum(axis=0, keepdims=True).sum(axis=1, keepdims=True)


MUTANTS = {
    "strided_head_mapping": ("kv_head_of", _m_strided_heads),
    "swapped_block_index": ("gather_sequence_kv", _m_swapped_block_index),
    "tail_off_by_one": ("gather_sequence_kv", _m_tail_off_by_one),
    "dropped_scale": ("attend", _m_no_scale),
    "normalise_by_length": ("attend", _m_divide_by_length),
    "wrong_logit_sign": ("attend", _m_wrong_sign),
    "softmax_over_heads": ("attend", _m_softmax_over_heads),
    "alibi_slope_dropped": ("alibi_bias", _m_alibi_slope_dropped),
    "alibi_wrong_head": ("alibi_bias", _m_alibi_wrong_head),
    "alibi_wrong_sign": ("alibi_bias", _m_alibi_sign),
}

PINS = [
    pins.test_hand_case_golden,
    lambda: pins.test_oracle_matches_brute_force(2, 6, 2, 16, 8, [9, 24], "bf16"),
    lambda: pins.test_oracle_matches_brute_force(3, 8, 1, 12, 16, [40, 17, 33], "fp16"),
    pins.test_single_token_returns_its_value_row,
    pins.test_identical_keys_give_mean_of_values,
    pins.test_hand_alibi_golden,
    lambda: pins.test_oracle_with_alibi_matches_brute_force(22, 8, 1, [33, 1, 12]),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setitem(pa.__dict__, "_orig_attend", pa.attend)
    monkeypatch.setitem(pa.__dict__, "_orig_alibi", pa.alibi_bias)
    monkeypatch.setattr(pa, attr, fn)
    caught = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError, FloatingPointError):
            caught += 1
    assert caught >= 1, f"no pin caught mutant {name}"


def test_unmutated_oracle_passes_every_pin():
    for pin in PINS:
        pin()
    assert math.isfinite(1.0)
