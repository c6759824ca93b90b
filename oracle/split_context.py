"""Split-context softmax: per-range partial results and their merge, float64.

The "Paged attention V2" column of the kernel-latency tables in
"[Performance] Support MQA/GQA in decode phase by using FlashAttention"
(vLLM pull request 2744) is named only; its numbers (about twice V1's speed
at batch 1, context 4096) fit the plain reading used here: the context is cut
into ranges, each range yields an unnormalised partial result, and a second
step merges them with a log-sum-exp weighting.

For a range R of tokens with logits x_t:
    m_R = max_{t in R} x_t
    l_R = sum_{t in R} exp(x_t - m_R)
    o_R = sum_{t in R} exp(x_t - m_R) * V[t]
and the merge over ranges is
    M = max_R m_R,  w_R = exp(m_R - M),
    out = (sum_R w_R o_R) / (sum_R w_R l_R),
which equals the unsplit softmax(x) @ V exactly in real arithmetic.
"""
from __future__ import annotations

import numpy as np


def partial(x, V):
    """(o_R, m_R, l_R) for logits x [n] and values V [n, D] of one range."""
    x = np.asarray(x, dtype=np.float64)
    m = float(x.max())
    w = np.exp(x - m)
    return w @ np.asarray(V, dtype=np.float64), m, float(w.sum())


def merge(parts):
    """Merge a list of (o_R, m_R, l_R) into the normalised output row."""
    M = max(m for _, m, _ in parts)
    num = sum(np.exp(m - M) * o for o, m, _ in parts)
    den = sum(np.exp(m - M) * l for _, m, l in parts)
    return num / den


def split_attention(x, V, bounds):
    """softmax(x) @ V computed as partials over [bounds[i], bounds[i+1]) ranges."""
    parts = [partial(x[a:b], V[a:b]) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    return merge(parts)
