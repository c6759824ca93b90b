"""gather_cached_kv: copy cached K/V rows at a slot mapping, bit for bit.

"Memcpy kernel for flash attention" (vLLM pull request 29) adds a kernel that
copies the cached keys and values of the tokens listed in a slot mapping into
contiguous [num_tokens, num_heads, head_size] tensors, so that an attention
kernel expecting contiguous K/V can consume them.  Its benchmark lines give
num_blocks and block_size alongside num_tokens; the plain reading of a slot is
``block_id * block_size + offset``, which is used here.

A slot outside [0, num_blocks * block_size) is invalid; its output row is all
zeros (a reading: the page does not say).
"""
from __future__ import annotations

import numpy as np


def gather_cached_kv(key_cache, value_cache, slot_mapping):
    """Return (key, value) arrays [T, H, D] with the same dtype as the caches."""
    NB, B = key_cache.shape[:2]
    slots = np.asarray(slot_mapping, dtype=np.int64)
    key = np.zeros((slots.size,) + key_cache.shape[2:], dtype=key_cache.dtype)
    value = np.zeros((slots.size,) + value_cache.shape[2:], dtype=value_cache.dtype)
    for t, slot in enumerate(slots.tolist()):
        if 0 <= slot < NB * B:
            key[t] = key_cache[slot // B, slot % B]
            value[t] = value_cache[slot // B, slot % B]
    return key, value
