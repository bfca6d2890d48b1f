"""Single-query paged GQA decode attention in float64 (test oracle).

What is computed, and where the pages say so:

* nano-vllm "Model Runner" notes, section "prefill and decode": at a decode
  step the query of the new token attends to all ``n`` K/V rows of its
  sequence (``n - 1`` cached plus the one stored this step).  ``context_len``
  is that ``n``.
* same notes, section "allocated kv cache": row ``j`` of sequence ``i`` is
  row ``j % block_size`` of physical block ``block_table[i][j // block_size]``
  of the per-layer cache ``[num_blocks, block_size, num_kv_heads, head_dim]``.
* Grok-1 "第 8 章 runners.py 推理引擎", section 8.5: 48 query heads share 8
  KV heads (grouped-query attention, ratio 6).  The pages do not spell out
  which query heads share a KV head; this oracle uses contiguous groups,
  query head ``h`` reads KV head ``h // (num_q_heads // num_kv_heads)``.
* Grok-1 section 8.2.3 (``hk_forward``): a row whose step is reset to 0
  attends to the empty set and its attention output is the zero vector.

* nanochat "04 · Engine 推理与工具调用", section "推理基准 infer_bench.py":
  a sliding-window layer reads only min(context, window) K/V rows.  The
  plainest reading, taken here: with a window W > 0 the query attends to the
  newest W positions of its context, [context_len - W, context_len) clipped
  at 0 (the new token included); W <= 0 means no window.

For each row i and query head h:
    s_j = scale * <q_{i,h}, K_j>        start_i <= j < context_len_i
    start_i = max(0, context_len_i - W) with a window W > 0, else 0
    p   = softmax(s)                    (max subtracted first)
    o   = sum_j p_j V_j
All arithmetic is float64 on exactly upcast inputs.
"""
from __future__ import annotations

import numpy as np


def gather_context(k_cache: np.ndarray, v_cache: np.ndarray, block_table,
                   context_len: int, kv_head: int):
    """K and V rows [context_len, D] of one sequence and KV head, in order."""
    block_size = k_cache.shape[1]
    ks, vs = [], []
    for j in range(int(context_len)):
        blk = int(block_table[j // block_size])
        row = j % block_size
        ks.append(k_cache[blk, row, kv_head])
        vs.append(v_cache[blk, row, kv_head])
    D = k_cache.shape[-1]
    if not ks:
        return np.zeros((0, D)), np.zeros((0, D))
    return np.asarray(ks, dtype=np.float64), np.asarray(vs, dtype=np.float64)


def attend(q_vec: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * K q) V for one query vector; zeros for an empty K."""
    q_vec = np.asarray(q_vec, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1] if V.ndim == 2 else q_vec.shape[-1])
    s = scale * (K @ q_vec)
    s = s - s.max()
    p = np.exp(s)
    p = p / p.sum()
    return p @ V


def window_start(context_len: int, window: int) -> int:
    """First attended position: the newest ``window`` of ``context_len`` (0 if no window)."""
    return max(0, int(context_len) - int(window)) if window and window > 0 else 0


def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     block_tables: np.ndarray, context_lens: np.ndarray,
                     scale: float, pairs=None, window: int = 0) -> np.ndarray:
    """Output [B, Hq, D] in float64 (or only the (row, head) ``pairs``).

    q: [B, Hq, D]; caches: [num_blocks, block_size, Hkv, D] (any float dtype,
    upcast exactly); block_tables: [B, max_blocks]; context_lens: [B];
    window > 0: attend to the newest ``window`` positions only.
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    if pairs is None:
        pairs = [(i, h) for i in range(B) for h in range(Hq)]
    cached = {}
    for i, h in pairs:
        hk = h // G
        key = (i, hk)
        if key not in cached:
            cached[key] = gather_context(k_cache, v_cache, block_tables[i],
                                         int(context_lens[i]), hk)
        K, V = cached[key]
        st = window_start(context_lens[i], window)
        K, V = K[st:], V[st:]
        out[i, h] = attend(q[i, h], K, V, scale) if K.shape[0] else 0.0
    return out


def partial_state(q_vec: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Unnormalised softmax state over a subset of the context.

    Returns (m, l, acc): m = max_j s_j, l = sum_j exp(s_j - m),
    acc = sum_j exp(s_j - m) V_j.
    """
    s = scale * (K @ np.asarray(q_vec, dtype=np.float64))
    m = s.max()
    w = np.exp(s - m)
    return m, w.sum(), w @ V


def lse_merge(states):
    """Combine partial states over disjoint parts of one context.

    M = max_s m_s,  L = sum_s l_s exp(m_s - M),
    o = sum_s exp(m_s - M) acc_s / L    (the softmax identity).
    """
    ms = np.array([s[0] for s in states], dtype=np.float64)
    ls = np.array([s[1] for s in states], dtype=np.float64)
    accs = np.array([s[2] for s in states], dtype=np.float64)
    M = ms.max()
    w = np.exp(ms - M)
    L = (w * ls).sum()
    return (w[:, None] * accs).sum(axis=0) / L
