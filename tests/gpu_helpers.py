"""Shared pieces of the GPU parity tests: building the library, moving the
seeded inputs to the device, and running the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

RAW = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}

# attention tolerances: fp32 max abs error; 16-bit relative per (row, head)
ATOL_F32 = 1e-4
RTOL_16 = 2e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_store_gb300 as pk
    return pk


def raw_numpy(t: torch.Tensor) -> np.ndarray:
    """Bit view of a host tensor as a numpy integer array (exact copy)."""
    return t.contiguous().view(RAW[t.dtype]).numpy().copy()


def from_raw(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(a).view(dtype)


def oracle_store_f64(w):
    """The oracle's store applied to the host workload; returns float64 K, V
    caches of the exercised layer and the oracle's slot mapping."""
    lay = w.layout
    slots = oracle.paging.decode_slot_mapping(lay.block_tables, lay.context_lens, w.cfg.block_size)
    k = raw_numpy(w.k_cache())
    v = raw_numpy(w.v_cache())
    oracle.store.kv_store(raw_numpy(w.k_new), raw_numpy(w.v_new), slots, k, v)
    kf = from_raw(k, w.cache.dtype).double().numpy()
    vf = from_raw(v, w.cache.dtype).double().numpy()
    return kf, vf, slots


def check_attention(out: np.ndarray, ref: np.ndarray, dtype: torch.dtype, pairs=None):
    """Assert the stated tolerance; returns the worst error seen."""
    if pairs is None:
        pairs = [(i, h) for i in range(ref.shape[0]) for h in range(ref.shape[1])]
    worst = 0.0
    for i, h in pairs:
        o, r = out[i, h], ref[i, h]
        assert np.all(np.isfinite(o)), (i, h, o)
        if dtype == torch.float32:
            e = float(np.abs(o - r).max())
            assert e <= ATOL_F32, (i, h, e)
        else:
            e = float(np.abs(o - r).max() / max(np.abs(r).max(), 1e-6))
            assert e <= RTOL_16, (i, h, e)
        worst = max(worst, e)
    return worst


def gather_rows_for_oracle(w, rows):
    """Blocks of the sampled rows copied to the host (before any kernel runs),
    with block tables remapped onto the copy.  Returns (k, v raw arrays,
    tables, the rows' context lengths)."""
    lay = w.layout
    bs = w.cfg.block_size
    blocks, tables = [], []
    for i in rows:
        n = -(-int(lay.context_lens[i]) // bs)
        ids = lay.block_tables[i, :n].tolist()
        tables.append(list(range(len(blocks), len(blocks) + n)) + [-1] * (lay.max_blocks_per_seq - n))
        blocks.extend(ids)
    idx = torch.tensor(blocks, dtype=torch.long, device=w.cache.device)
    k = w.cache[0, lay.layer].index_select(0, idx).cpu()
    v = w.cache[1, lay.layer].index_select(0, idx).cpu()
    return raw_numpy(k), raw_numpy(v), np.array(tables, dtype=np.int64), lay.context_lens[rows]


def oracle_sampled(w, gathered, rows, heads_per_row, window=0):
    """Oracle attention for sampled (row, head) pairs of a device workload."""
    k, v, tables, ctx = gathered
    bs = w.cfg.block_size
    sub_slots = oracle.paging.decode_slot_mapping(tables, ctx, bs)
    k_new = raw_numpy(w.k_new[rows].cpu())
    v_new = raw_numpy(w.v_new[rows].cpu())
    oracle.store.kv_store(k_new, v_new, sub_slots, k, v)
    dt = w.cache.dtype
    kf = from_raw(k, dt).double().numpy()
    vf = from_raw(v, dt).double().numpy()
    q = w.q[rows].cpu().double().numpy()
    pairs = [(r, h) for r in range(len(rows)) for h in heads_per_row]
    return oracle.attention.decode_attention(q, kf, vf, tables, ctx, w.scale, pairs=pairs, window=window), pairs
