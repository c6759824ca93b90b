"""Write new tokens' K/V into the paged pool at a slot mapping (bit copy).

The notes of "[Performance] Support MQA/GQA in decode phase by using
FlashAttention" (vLLM pull request 2744) name ``cache_ops.cache``: the step
that stores each new token's key and value into its cache slot before decode
attention reads them.  It is the inverse of gather_cached_kv.  A slot is
``block_id * block_size + offset``; a negative slot marks a token that is not
stored (a reading: padding tokens), and a slot at or past
num_blocks * block_size is invalid and not stored either.
"""
from __future__ import annotations

import numpy as np


def cache_kv(key, value, key_cache, value_cache, slot_mapping):
    """Return updated copies of (key_cache, value_cache)."""
    kc = np.array(key_cache, copy=True)
    vc = np.array(value_cache, copy=True)
    NB, B = kc.shape[:2]
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64).tolist()):
        if 0 <= slot < NB * B:
            kc[slot // B, slot % B] = key[t]
            vc[slot // B, slot % B] = value[t]
    return kc, vc
