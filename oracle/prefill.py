"""Varlen paged prefill: slot mapping, store and causal attention (test oracle).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.

What is computed, and where the pages say so:

* nano-vllm "Model Runner" notes, section "prefix cache": a prefill batch is
  described by ``cu_seqlens_q`` (prefix sums of the tokens scheduled for each
  sequence now) and ``cu_seqlens_k`` (prefix sums of scheduled plus already
  cached tokens); a batch has prefix-cache hits exactly when
  ``cu_seqlens_k[-1] > cu_seqlens_q[-1]``.
* same notes, section "prepare Prefill": the block table is filled by the
  scheduler before the step; the step derives each new token's slot from it
  and the attention layer writes the new K/V rows to those slots.
* same notes, section "prefill and decode": prefill computes the K/V of all
  scheduled tokens at once (a dense, compute-bound step); decode is the
  one-token case of the same bookkeeping.
* same notes, section "allocated kv cache": slot arithmetic (see ``paging``).

Readings where the pages leave a step open (plainest choice):

* Sequence i has ``q_i = cu_q[i+1] - cu_q[i]`` new tokens and
  ``k_i = cu_k[i+1] - cu_k[i]`` tokens in all, ``k_i >= q_i``; its first
  ``c_i = k_i - q_i`` positions are the cached prefix, so new token j sits at
  position ``c_i + j``.
* Causal attention: the new token at position p attends to positions
  ``0 .. p`` of its own sequence (the cached prefix, the earlier new tokens
  and itself), read through the block table after this step's store.
* The sliding window of the decode path carries over: with W > 0 the token at
  position p attends to ``[max(0, p + 1 - W), p]``; W <= 0 means no window.
* Chunked prefill is the same computation: an earlier chunk is a cached
  prefix of the next.

All floating-point arithmetic is float64 on exactly upcast inputs.
"""
from __future__ import annotations

import numpy as np

from .attention import attend, gather_context, window_start
from .paging import slot_of_position


def sequence_lengths(cu_seqlens_q, cu_seqlens_k):
    """(q_lens, k_lens, cached_lens) as int64 arrays; checks the shapes."""
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    if cq.ndim != 1 or cq.shape != ck.shape or len(cq) < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be 1-D of equal length >= 1")
    if cq[0] != 0 or ck[0] != 0:
        raise ValueError("cu_seqlens must start at 0")
    q_lens = np.diff(cq)
    k_lens = np.diff(ck)
    if (q_lens < 0).any() or (k_lens < q_lens).any():
        raise ValueError("need 0 <= q_len <= k_len for every sequence")
    return q_lens, k_lens, k_lens - q_lens


def has_prefix_hits(cu_seqlens_q, cu_seqlens_k) -> bool:
    """The pages' test for a batch with cached prefixes."""
    return int(cu_seqlens_k[-1]) > int(cu_seqlens_q[-1])


def token_positions(cu_seqlens_q, cu_seqlens_k):
    """For each new token t (in cu_seqlens_q order): (sequence, position)."""
    q_lens, _, cached = sequence_lengths(cu_seqlens_q, cu_seqlens_k)
    seq, pos = [], []
    for i in range(len(q_lens)):
        for j in range(int(q_lens[i])):
            seq.append(i)
            pos.append(int(cached[i]) + j)
    return np.asarray(seq, dtype=np.int64), np.asarray(pos, dtype=np.int64)


def prefill_slot_mapping(block_tables: np.ndarray, cu_seqlens_q, cu_seqlens_k,
                         block_size: int) -> np.ndarray:
    """Slot of every new token, int64 [total_q] (cu_seqlens_q order)."""
    seq, pos = token_positions(cu_seqlens_q, cu_seqlens_k)
    out = np.empty(len(seq), dtype=np.int64)
    for t in range(len(seq)):
        out[t] = slot_of_position(block_tables[seq[t]], int(pos[t]), block_size)
    return out


def prefill_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      block_tables: np.ndarray, cu_seqlens_q, cu_seqlens_k,
                      scale: float, window: int = 0, pairs=None) -> np.ndarray:
    """Output [total_q, Hq, D] in float64 (or only the (token, head) ``pairs``).

    q: [total_q, Hq, D]; caches: [num_blocks, block_size, Hkv, D] holding
    every sequence's rows 0 .. k_len-1 (the new rows already stored);
    block_tables: [num_seqs, max_blocks]; query head h reads KV head
    h // (Hq // Hkv) (contiguous groups, as in the decode oracle).
    """
    T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    _, k_lens, _ = sequence_lengths(cu_seqlens_q, cu_seqlens_k)
    seq, pos = token_positions(cu_seqlens_q, cu_seqlens_k)
    if len(seq) != T:
        raise ValueError("q rows must equal cu_seqlens_q[-1]")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    if pairs is None:
        pairs = [(t, h) for t in range(T) for h in range(Hq)]
    ctx = {}
    for t, h in pairs:
        i, p = int(seq[t]), int(pos[t])
        key = (i, h // G)
        if key not in ctx:
            ctx[key] = gather_context(k_cache, v_cache, block_tables[i], int(k_lens[i]), h // G)
        K, V = ctx[key]
        st = window_start(p + 1, window)
        out[t, h] = attend(q[t, h], K[st:p + 1], V[st:p + 1], scale)
    return out

