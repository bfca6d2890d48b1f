"""GB300 paged-KV decode step: Python binding of the libpkvd C ABI.

The functions below only marshal torch tensors into the C calls declared in
``include/pkvd.h``; every step of the decode path runs in the library's CUDA
kernels.  If ``libpkvd.so`` has not been built, every call raises.

    slot_mapping(block_tables, context_lens, block_size, num_blocks)
    kv_store(k, v, slot_mapping, k_cache, v_cache)
    paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, scale)
    sample(logits, temperature, top_k, top_p, seeds, offsets)
    DecodeStep(...)   -- the four calls captured in one CUDA graph
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._capi import (LIB_PATH, PATH_AUTO, PATH_FMA, PATH_MMA, PATH_TC, ERR_BLOCK_ID, ERR_SLOT,  # noqa: F401
                    ERR_CONTEXT, ERR_TIMEOUT, PkvdCache, PkvdError, lib, check, dtype_code,
                    stream_handle, cache_desc, ptr)
from .step import DecodeStep  # noqa: F401
from .block_manager import BlockManager, shared_prefix_len  # noqa: F401

__all__ = ["BlockManager", "copy_blocks", "slot_mapping", "kv_store", "kv_store_paged", "kv_store_prefill",
           "prefill_attention", "sample_ex", "pack_mask", "paged_decode_attention", "decode_workspace_bytes",
           "paged_decode_attention_prefix", "decode_prefix_workspace_bytes", "shared_prefix_len",
           "sample", "DecodeStep", "PkvdError", "lib"]


def _err_ptr(err):
    return ptr(err) if err is not None else None


def slot_mapping(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int,
                 num_blocks: int, out: torch.Tensor | None = None, err: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """int64 slot of each row's new token (-1 for an empty row)."""
    B = context_lens.shape[0]
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=context_lens.device)
    check(lib().pkvd_slot_mapping(ptr(out), ptr(block_tables), block_tables.shape[1],
                                  ptr(context_lens), B, block_size, num_blocks,
                                  stream_handle(stream, out), _err_ptr(err)))
    return out


def kv_store(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor, err: torch.Tensor | None = None,
             stream=None) -> None:
    """Write k[i], v[i] ([N, Hkv, D], contiguous) into slot_mapping[i] of the caches
    ([num_blocks, block_size, Hkv, D] views, modified in place)."""
    c = cache_desc(k_cache, v_cache)
    check(lib().pkvd_kv_store(ptr(k), ptr(v), ptr(slot_mapping), k.shape[0], ctypes.byref(c),
                              stream_handle(stream, k), _err_ptr(err)))


def kv_store_paged(k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor | None = None,
                   err: torch.Tensor | None = None, stream=None) -> None:
    """Slot mapping and store in one kernel: row i's k[i], v[i] go to the slot of
    its newest token (context_lens[i] - 1 through block_tables[i]); the slots are
    also written to slot_mapping (int64 [B]) when it is given."""
    c = cache_desc(k_cache, v_cache)
    check(lib().pkvd_kv_store_paged(ptr(k), ptr(v), ptr(block_tables), block_tables.shape[1],
                                    ptr(context_lens), k.shape[0], ptr(slot_mapping), ctypes.byref(c),
                                    stream_handle(stream, k), _err_ptr(err)))


def kv_store_prefill(k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor, cu_seqlens_q: torch.Tensor,
                     cu_seqlens_k: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     slot_mapping: torch.Tensor | None = None, err: torch.Tensor | None = None,
                     stream=None) -> None:
    """Varlen prefill store: new row t of sequence i (rows cu_seqlens_q[i] ..
    cu_seqlens_q[i+1]-1) goes to the slot of position (k_len_i - q_len_i) +
    (t - cu_seqlens_q[i]); the slots are also written to slot_mapping (int64
    [total_q]) when it is given."""
    c = cache_desc(k_cache, v_cache)
    check(lib().pkvd_kv_store_prefill(ptr(k), ptr(v), ptr(block_tables), block_tables.shape[1],
                                      ptr(cu_seqlens_q), ptr(cu_seqlens_k), cu_seqlens_q.shape[0] - 1,
                                      k.shape[0], ptr(slot_mapping), ctypes.byref(c),
                                      stream_handle(stream, k), _err_ptr(err)))


def prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                      max_seqlen_q: int, scale: float, window: int = 0, out: torch.Tensor | None = None,
                      err: torch.Tensor | None = None, stream=None, path: int = PATH_AUTO) -> torch.Tensor:
    """Causal varlen attention of the new rows q ([total_q, Hq, D]) over their
    sequences' cached prefix and new rows, read from the paged cache
    (path: PATH_AUTO, PATH_TC for tcgen05, PATH_MMA for mma.sync)."""
    T, Hq, _ = q.shape
    c = cache_desc(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    check(lib().pkvd_prefill_attention_ex(ptr(out), ptr(q), ctypes.byref(c), ptr(block_tables),
                                          block_tables.shape[1], ptr(cu_seqlens_q), ptr(cu_seqlens_k),
                                          cu_seqlens_q.shape[0] - 1, T, max_seqlen_q, Hq,
                                          ctypes.c_float(scale), window, stream_handle(stream, q), _err_ptr(err),
                                          path))
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src: torch.Tensor, dst: torch.Tensor,
                rows: torch.Tensor, err: torch.Tensor | None = None, stream=None) -> None:
    """Copy-on-write: the first rows[i] token rows of block src[i] -> block dst[i]
    (K and V; src, dst, rows: int32 device tensors)."""
    c = cache_desc(k_cache, v_cache)
    check(lib().pkvd_copy_blocks(ctypes.byref(c), ptr(src), ptr(dst), ptr(rows), src.numel(),
                                 stream_handle(stream, k_cache), _err_ptr(err)))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                           sm_count: int = 0) -> int:
    n = ctypes.c_size_t(0)
    check(lib().pkvd_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                            sm_count, ctypes.byref(n)))
    return int(n.value)


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           max_context_len: int, scale: float, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, err: torch.Tensor | None = None,
                           stream=None, path: int = PATH_AUTO, window: int = 0) -> torch.Tensor:
    """out[i, h] = softmax(scale * q[i, h] . K_i^T) V_i over row i's paged context
    (its newest `window` positions when window > 0)."""
    B, Hq, D = q.shape
    c = cache_desc(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = decode_workspace_bytes(B, Hq, D, max_context_len)
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if window:
        check(lib().pkvd_paged_decode_attention_window(
            ptr(out), ptr(q), ctypes.byref(c), ptr(block_tables), block_tables.shape[1],
            ptr(context_lens), max_context_len, B, Hq, ctypes.c_float(scale), window, ptr(workspace),
            workspace.numel() * workspace.element_size(), stream_handle(stream, q), _err_ptr(err), path))
        return out
    check(lib().pkvd_paged_decode_attention_ex(
        ptr(out), ptr(q), ctypes.byref(c), ptr(block_tables), block_tables.shape[1],
        ptr(context_lens), max_context_len, B, Hq, ctypes.c_float(scale), ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream, q), _err_ptr(err), path))
    return out


def decode_prefix_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                  max_context_len: int, prefix_len: int, sm_count: int = 0) -> int:
    n = ctypes.c_size_t(0)
    check(lib().pkvd_decode_prefix_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                                   prefix_len, sm_count, ctypes.byref(n)))
    return int(n.value)


def paged_decode_attention_prefix(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  max_context_len: int, scale: float, prefix_len: int,
                                  out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                  err: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_decode_attention for rows whose first prefix_len cached tokens are
    the same blocks in every row's table (read once per group of rows)."""
    B, Hq, D = q.shape
    c = cache_desc(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = decode_prefix_workspace_bytes(B, Hq, k_cache.shape[2], D, max_context_len, prefix_len)
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    check(lib().pkvd_paged_decode_attention_prefix(
        ptr(out), ptr(q), ctypes.byref(c), ptr(block_tables), block_tables.shape[1], ptr(context_lens),
        max_context_len, B, Hq, ctypes.c_float(scale), prefix_len, ptr(workspace),
        workspace.numel() * workspace.element_size(), stream_handle(stream, q), _err_ptr(err)))
    return out


def sample(logits: torch.Tensor, temperature: torch.Tensor, top_k: torch.Tensor,
           top_p: torch.Tensor, seeds: torch.Tensor, offsets: torch.Tensor,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int32 token id per row: temperature, top-k, nucleus cut, Philox Gumbel-max."""
    R, V = logits.shape
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    if out is None:
        out = torch.empty(R, dtype=torch.int32, device=logits.device)
    check(lib().pkvd_sample(ptr(out), ptr(logits), dtype_code(logits.dtype), R, V, logits.stride(0),
                            ptr(temperature), ptr(top_k), ptr(top_p), ptr(seeds), ptr(offsets),
                            None, 0, stream_handle(stream, logits)))
    return out



def pack_mask(allowed: torch.Tensor) -> torch.Tensor:
    """Bool [R, V] (True = may be drawn) -> the int32 [R, ceil(V/32)] bit words
    pkvd_sample_ex takes (bit j % 32 of word j / 32)."""
    R, V = allowed.shape
    W = (V + 31) // 32
    bits = torch.zeros(R, W * 32, dtype=torch.int64, device=allowed.device)
    bits[:, :V] = allowed.to(torch.int64)
    weights = torch.pow(2, torch.arange(32, device=allowed.device, dtype=torch.int64))
    words = (bits.view(R, W, 32) * weights).sum(-1)
    return torch.where(words >= 2**31, words - 2**32, words).to(torch.int32)


def sample_ex(logits: torch.Tensor, temperature: torch.Tensor, top_k: torch.Tensor, top_p: torch.Tensor,
              seeds: torch.Tensor, offsets: torch.Tensor, mask_words: torch.Tensor | None = None,
              with_probs: bool = True, stream=None):
    """sample() plus Grok's extras: an optional allowed-id bit mask (pack_mask),
    and (with_probs) the drawn token's probability and the top-8 probabilities
    and ids.  Returns (token_ids, token_prob, top_probs, top_ids)."""
    R, V = logits.shape
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    dev = logits.device
    out = torch.empty(R, dtype=torch.int32, device=dev)
    tp = torch.empty(R, dtype=torch.float32, device=dev) if with_probs else None
    p8 = torch.empty(R, 8, dtype=torch.float32, device=dev) if with_probs else None
    i8 = torch.empty(R, 8, dtype=torch.int32, device=dev) if with_probs else None
    n = ctypes.c_size_t(0)
    check(lib().pkvd_sample_workspace_bytes(R, V, ctypes.byref(n)))
    ws = torch.empty(max(int(n.value), 16), dtype=torch.uint8, device=dev)
    mw = mask_words.shape[1] if mask_words is not None else 0
    check(lib().pkvd_sample_ex(ptr(out), ptr(logits), dtype_code(logits.dtype), R, V, logits.stride(0),
                               ptr(temperature), ptr(top_k), ptr(top_p), ptr(seeds), ptr(offsets),
                               ptr(mask_words), mw, ptr(tp), ptr(p8), ptr(i8), ptr(ws), ws.numel(),
                               stream_handle(stream, logits)))
    return out, tp, p8, i8