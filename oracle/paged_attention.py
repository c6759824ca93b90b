"""Decode-phase attention over a paged KV cache, float64, by its definition.

The operation is the one vLLM calls ``single_query_cached_kv_attention``
("Optimizes the single_query_cached_kv_attention kernel", vLLM pull request
420): each sequence contributes ONE new query token per head, which attends
over every token already in that sequence's KV cache.  The pages describe the
kernel but print no formula; the plain reading, used here, is

    out[s, h, :] = softmax_t(scale * q[s, h, :] . K_s[t, :]) @ V_s[t, :]

over t < context_lens[s], with

    K_s[t] = key_cache[block_tables[s, t // B], t % B, kv(h), :]   (V alike)

for cache tensors laid out [num_blocks, block_size B, num_kv_heads, head_size].

Query head h reads KV head kv(h) = h // (num_heads // num_kv_heads): the
review suggestion on "Optimize MQA Kernel" (vLLM pull request 452) builds the
head mapping as ``repeat_interleave(arange(num_kv_heads), num_queries_per_kv)``
after asserting ``num_heads % num_kv_heads == 0``, i.e. contiguous groups of
query heads share one KV head.  num_kv_heads == num_heads is MHA, 1 is MQA,
anything between is GQA.

ALiBi (optional): "Optimize MQA Kernel" notes that MQA combines with ALiBi
embeddings, and the kernel-latency runs of "[Performance] Support MQA/GQA in
decode phase by using FlashAttention" are made with use_alibi=False.  The
plain reading of ALiBi for the single decode query (position L - 1) adds a
per-head linear bias to each logit:

    logit[s, h, t] = scale * q . K_s[t] + slopes[h] * (t - L + 1)

Readings of what the pages leave open (also listed in the design notes):
  * context_lens[s] == 0 gives an all-zero output row;
  * a sequence whose length is negative, exceeds the table
    (max_blocks_per_seq * B) or exceeds the caller's ``max_context_len``, or
    whose referenced block ids fall outside [0, num_blocks), is invalid and
    its output is all zeros;
  * table entries past ceil(L / B) and cache slots past L are never read.

The softmax subtracts the row maximum before exponentiating; this changes no
value mathematically and keeps float64 from overflowing.
"""
from __future__ import annotations

import numpy as np

from .formats import decode_bits


def kv_head_of(h: int, num_heads: int, num_kv_heads: int) -> int:
    """KV head read by query head h (contiguous groups of query heads)."""
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    return h // (num_heads // num_kv_heads)


def sequence_is_valid(block_tables, context_lens, s: int, block_size: int, num_blocks: int,
                      max_context_len: int | None = None) -> bool:
    L = int(context_lens[s])
    mb = block_tables.shape[1]
    if L < 0 or L > mb * block_size:
        return False
    if max_context_len is not None and L > max_context_len:
        return False
    ids = np.asarray(block_tables[s, : -(-L // block_size)], dtype=np.int64)
    return bool(np.all((ids >= 0) & (ids < num_blocks)))


def gather_sequence_kv(cache_bits, block_tables, s: int, L: int, kv: int, dtype: str):
    """Rows t < L of KV head ``kv`` for sequence s, through the block table."""
    B = cache_bits.shape[1]
    t = np.arange(L)
    phys = np.asarray(block_tables[s], dtype=np.int64)[t // B]
    return decode_bits(cache_bits[phys, t % B, kv, :], dtype)


def attend(Q, K, V, scale: float, bias=None):
    """softmax over tokens of scale * Q K^T (+ bias [n, L]), times V.
    Q [n, D], K/V [L, D] -> [n, D]."""
    X = float(scale) * (Q @ K.T)                          # [n, L]
    if bias is not None:
        X = X + bias
    X = X - X.max(axis=1, keepdims=True)
    P = np.exp(X)
    return (P @ V) / P.sum(axis=1, keepdims=True)


def alibi_bias(slopes, heads, L: int):
    """Bias [len(heads), L] = slopes[h] * (t - L + 1)."""
    t = np.arange(L, dtype=np.float64) - (L - 1)
    return np.asarray(slopes, dtype=np.float64)[list(heads)][:, None] * t[None, :]


def paged_decode_attention(q, key_cache, value_cache, block_tables, context_lens, scale: float,
                           dtype: str, *, pairs=None, max_context_len: int | None = None,
                           alibi_slopes=None):
    """Reference decode attention.

    q: uint16 bits [S, H, D]; key_cache / value_cache: uint16 bits
    [NB, B, Hk, D]; block_tables: int [S, MB]; context_lens: int [S].
    alibi_slopes: optional float [H] ALiBi slopes.
    Returns float64 [S, H, D], or [len(pairs), D] for a list of (s, h) pairs.
    """
    S, H, D = q.shape
    NB, B, Hk, _ = key_cache.shape
    g = H // Hk
    if H % Hk:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    if pairs is None:
        want = {s: list(range(H)) for s in range(S)}
    else:
        want = {}
        for s, h in pairs:
            want.setdefault(int(s), []).append(int(h))
    res = {}
    for s, heads in want.items():
        valid = sequence_is_valid(block_tables, context_lens, s, B, NB, max_context_len)
        L = int(context_lens[s])
        by_kv = {}
        for h in heads:
            by_kv.setdefault(kv_head_of(h, H, Hk), []).append(h)
        for kv, hs in by_kv.items():
            if not valid or L == 0:
                for h in hs:
                    res[(s, h)] = np.zeros(D)
                continue
            K = gather_sequence_kv(key_cache, block_tables, s, L, kv, dtype)
            V = gather_sequence_kv(value_cache, block_tables, s, L, kv, dtype)
            bias = None if alibi_slopes is None else alibi_bias(alibi_slopes, hs, L)
            O = attend(decode_bits(q[s, hs, :], dtype), K, V, scale, bias)
            for i, h in enumerate(hs):
                res[(s, h)] = O[i]
    if pairs is None:
        out = np.zeros((S, H, D))
        for (s, h), v in res.items():
            out[s, h] = v
        return out
    return np.stack([res[(int(s), int(h))] for s, h in pairs]) if len(pairs) else np.zeros((0, D))
