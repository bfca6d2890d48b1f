"""Slot arithmetic and KV-cache sizing (test oracle; float-free integer math).

Sources:
* nano-vllm "Model Runner" notes, section "allocated kv cache": the cache is
  ``[2, num_layers, num_blocks, block_size, num_kv_heads, head_dim]``; a
  token at position ``pos`` of a sequence lives in logical block
  ``pos // block_size``, physical block ``block_table[logical]``, row
  ``pos % block_size``, i.e. slot ``physical * block_size + pos % block_size``;
  one physical block across all layers costs
  ``2 * num_layers * block_size * num_kv_heads * head_dim * itemsize`` bytes.
* same notes, section "prefill and decode": at a decode step with ``n``
  tokens, ``n - 1`` K/V rows are already cached and the n-th is computed and
  stored now, so the new token's position is ``context_len - 1``.
* Grok-1 "第 8 章 runners.py 推理引擎", section 8.5: a contiguous per-layer
  cache of ``[B, T, num_kv_heads, head_dim]`` for k and for v.
"""
from __future__ import annotations

import numpy as np


def slot_of_position(block_table, position: int, block_size: int) -> int:
    """Flat slot index of token ``position`` of one sequence."""
    logical = position // block_size
    physical = int(block_table[logical])
    return physical * block_size + position % block_size


def decode_slot_mapping(block_tables: np.ndarray, context_lens: np.ndarray,
                        block_size: int) -> np.ndarray:
    """Slot of each row's new token; -1 marks an inactive row (context 0)."""
    B = len(context_lens)
    out = np.full(B, -1, dtype=np.int64)
    for i in range(B):
        ctx = int(context_lens[i])
        if ctx > 0:
            out[i] = slot_of_position(block_tables[i], ctx - 1, block_size)
    return out


def paged_block_bytes(num_layers: int, block_size: int, num_kv_heads: int,
                      head_dim: int, itemsize: int) -> int:
    """Bytes one physical block occupies across K and V of every layer."""
    return 2 * num_layers * block_size * num_kv_heads * head_dim * itemsize


def contiguous_cache_bytes(num_layers: int, max_len: int, num_kv_heads: int,
                           head_dim: int, itemsize: int, batch: int = 1) -> int:
    """Bytes of a max_len-preallocated K and V cache for every layer."""
    return num_layers * 2 * batch * max_len * num_kv_heads * head_dim * itemsize


def blocks_needed(context_len: int, block_size: int) -> int:
    """Physical blocks a sequence of ``context_len`` tokens occupies."""
    return -(-int(context_len) // block_size)
