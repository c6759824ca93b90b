"""Dense decode attention by triple loop, pure Python floats (tiny inputs).

Independent of the paged oracle: it takes one query vector and contiguous
lists of key and value rows, and evaluates softmax(scale * q . k_t) @ V with
nothing but ``math.exp`` and Python float (binary64) arithmetic.
"""
from __future__ import annotations

import math


def dense_decode_attention(q, K, V, scale, alibi_slope=0.0):
    """q: [D] floats; K, V: [L][D] floats; returns [D] floats (zeros if L == 0).
    alibi_slope adds slope * (t - L + 1) to the logit of token t."""
    D = len(q)
    L = len(K)
    if L == 0:
        return [0.0] * D
    logits = []
    for t in range(L):
        acc = 0.0
        for d in range(D):
            acc += q[d] * K[t][d]
        logits.append(scale * acc + alibi_slope * (t - (L - 1)))
    top = max(logits)
    weights = [math.exp(x - top) for x in logits]
    total = math.fsum(weights)
    out = []
    for d in range(D):
        out.append(math.fsum(weights[t] * V[t][d] for t in range(L)) / total)
    return out
