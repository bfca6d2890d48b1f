"""Scalar KV-cache store through ``slot_mapping`` (test oracle).

nano-vllm "Model Runner" notes, sections "prepare Prefill" and "allocated kv
cache": the attention layer writes each new token's K and V to its slot of
the per-layer cache ``[num_blocks, block_size, num_kv_heads, head_dim]``
(K = ``kv_cache[0, layer]``, V = ``kv_cache[1, layer]``).  Grok-1 section 8.5
(donated buffers) makes the update in place.  The copy is exact: the bits of
each element are moved, nothing is converted.

A negative slot marks a padded or inactive row and is skipped (the inactive
rows of Grok-1 section 8.2.3 take part in the step but their results are not
used).
"""
from __future__ import annotations

import numpy as np


def kv_store(k_new: np.ndarray, v_new: np.ndarray, slot_mapping: np.ndarray,
             k_cache: np.ndarray, v_cache: np.ndarray) -> None:
    """Copy row i of k_new / v_new ([N, Hkv, D]) into slot_mapping[i].

    The caches are modified in place.  Arrays may hold raw integer views of
    16-bit floats; the copy never looks at values.
    """
    num_blocks, block_size = k_cache.shape[0], k_cache.shape[1]
    seen = set()
    for i in range(len(slot_mapping)):
        slot = int(slot_mapping[i])
        if slot < 0:
            continue
        if slot >= num_blocks * block_size:
            raise IndexError(f"slot {slot} outside the cache")
        if slot in seen:
            raise ValueError(f"slot {slot} written twice in one step")
        seen.add(slot)
        blk, row = divmod(slot, block_size)
        k_cache[blk, row] = k_new[i]
        v_cache[blk, row] = v_new[i]
