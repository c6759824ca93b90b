"""Prefill (a chunk of several new query tokens per sequence) over a paged KV
cache, float64, by its definition.  TEST INFRASTRUCTURE ONLY (see the package
header).

Source: the review comments on "[Performance] Support MQA/GQA in decode phase
by using FlashAttention" (vLLM pull request 2744) note that the kernel which
attends new queries over the paged KV cache (flash-attn's
``flash_attn_with_kvcache``) serves prefill as well, both without and with a
cached prefix.  The page prints no formula.  The plain reading, used here:

A sequence s brings a chunk of n_s new tokens whose K/V rows were already
written into its paged cache as its LAST n_s tokens, so context_lens[s] = L_s
counts them (with n_s = L_s there is no prefix).  Query i of the chunk
(0 <= i < n_s) sits at position p = L_s - n_s + i and attends causally to the
cache tokens up to and including its own position:

    out[q0_s + i, h, :] = softmax_{t <= p}(scale * q[q0_s + i, h, :] . K_s[t, :]) @ V_s[t, :]

with q and out packed token-major [sum_s n_s, H, D], q0_s = query_start[s]
(query_start[S] = sum_s n_s), K_s / V_s read through the block table exactly
as for decode, and the same contiguous query-head -> KV-head groups.  n_s = 1
is decode.  With ALiBi the logit of token t for query i gains
slopes[h] * (t - p): the decode bias taken at the query's own position.

Readings of what the page leaves open (also listed in the design notes):
  * n_s = 0 contributes no rows;
  * a sequence with n_s > L_s, a negative length, a length longer than its
    table or than max_context_len, or a chunk longer than max_query_len is
    invalid: all its query rows are zeros;
  * a query whose window t <= p references a block id outside
    [0, num_blocks) gives a zero row; queries before the bad block are
    unaffected (for decode the window is the whole sequence, so this is the
    decode rule).
"""
from __future__ import annotations

import numpy as np

from .formats import decode_bits
from .paged_attention import alibi_bias, attend, gather_sequence_kv, kv_head_of


def query_position(L: int, n: int, i: int) -> int:
    """Position in the sequence of query i of a chunk of n ending at length L."""
    return L - n + i


def visible_tokens(p: int) -> int:
    """Number of cache tokens a query at position p attends to (t <= p)."""
    return p + 1


def paged_prefill_attention(q, key_cache, value_cache, block_tables, context_lens, query_start,
                            scale: float, dtype: str, *, max_context_len: int | None = None,
                            max_query_len: int | None = None, alibi_slopes=None, rows=None):
    """Reference prefill attention.

    q: uint16 bits [T, H, D] (T = query_start[-1]); key_cache / value_cache:
    uint16 bits [NB, B, Hk, D]; block_tables: int [S, MB]; context_lens: int
    [S]; query_start: int [S + 1], non-decreasing from 0.  Returns float64
    [T, H, D], or [len(rows), D] for a list of (token row, head) pairs.
    """
    T, H, D = q.shape
    NB, B, Hk, _ = key_cache.shape
    S = len(context_lens)
    qs = np.asarray(query_start, dtype=np.int64)
    if qs.shape != (S + 1,) or qs[0] != 0 or qs[-1] != T or np.any(np.diff(qs) < 0):
        raise ValueError("query_start must be [S + 1], non-decreasing from 0 to T")
    want = None
    if rows is not None:
        want = {}
        for r, h in rows:
            want.setdefault(int(r), set()).add(int(h))
    res = {}
    for s in range(S):
        n = int(qs[s + 1] - qs[s])
        if n == 0:
            continue
        L = int(context_lens[s])
        length_ok = (0 <= L <= block_tables.shape[1] * B and n <= L and
                     (max_context_len is None or L <= max_context_len) and
                     (max_query_len is None or n <= max_query_len))
        seq_rows = range(int(qs[s]), int(qs[s + 1]))
        if want is not None:
            seq_rows = [r for r in seq_rows if r in want]
        if not length_ok:
            for r in seq_rows:
                for h in range(H):
                    res[(r, h)] = np.zeros(D)
            continue
        # First token whose block id is out of range (L if none).
        ids = np.asarray(block_tables[s, : -(-L // B)], dtype=np.int64)
        bad = np.nonzero((ids < 0) | (ids >= NB))[0]
        first_bad = int(bad[0]) * B if bad.size else L
        for kv in range(Hk):
            hs = [h for h in range(H) if kv_head_of(h, H, Hk) == kv]
            K = V = None
            for r in seq_rows:
                heads = hs if want is None else [h for h in hs if h in want[r]]
                if not heads:
                    continue
                p = query_position(L, n, r - int(qs[s]))
                nv = visible_tokens(p)
                if nv > first_bad:
                    for h in heads:
                        res[(r, h)] = np.zeros(D)
                    continue
                if K is None:
                    K = gather_sequence_kv(key_cache, block_tables, s, first_bad, kv, dtype)
                    V = gather_sequence_kv(value_cache, block_tables, s, first_bad, kv, dtype)
                bias = None if alibi_slopes is None else alibi_bias(alibi_slopes, heads, nv)
                O = attend(decode_bits(q[r, heads, :], dtype), K[:nv], V[:nv], scale, bias)
                for k, h in enumerate(heads):
                    res[(r, h)] = O[k]
    if rows is None:
        out = np.zeros((T, H, D))
        for (r, h), v in res.items():
            out[r, h] = v
        return out
    return (np.stack([res.get((int(r), int(h)), np.zeros(D)) for r, h in rows])
            if len(rows) else np.zeros((0, D)))
