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


def sampling_exempt(info, p):
    """True where float rounding may decide the draw: the oracle's two best
    perturbed scores closer than 1e-5 * max(1, |s1|), or the nucleus cut mass
    within 1e-6 of p (the readings of the "< 1e-5" rule and of the boundary)."""
    if info["top2_gap"] < 1e-5 * max(1.0, abs(info["top1_score"])):
        return True
    n = info["nucleus"]
    if n is not None and (abs(n["mass_before"] - p) < 1e-6 or abs(n["mass_after"] - p) < 1e-6):
        return True
    return False


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


def oracle_rows_by_kv_head(w, rows, kv_heads_of_row):
    """Oracle attention of whole rows of a (device) workload, for the listed KV
    heads of each row and all their query heads.

    Each row's blocks, restricted to those KV heads, are copied off the device
    into a small cache of their own (call this before any kernel stores into
    the cache); the oracle's store then writes the row's new token there and
    the oracle's attention runs on it.  Returns {row: (query heads, output
    [len(query heads), D] float64)}."""
    lay, cfg = w.layout, w.cfg
    bs, G, dt = cfg.block_size, cfg.group, w.cache.dtype
    kc, vc = w.cache[0, lay.layer], w.cache[1, lay.layer]
    res = {}
    for i in rows:
        c = int(lay.context_lens[i])
        n = -(-c // bs)
        hks = list(kv_heads_of_row[i])
        heads = [hk * G + g for hk in hks for g in range(G)]
        if n == 0:
            res[i] = (heads, np.zeros((len(heads), cfg.head_dim)))
            continue
        idx = torch.from_numpy(lay.block_tables[i, :n].astype(np.int64)).to(kc.device)
        hsel = torch.tensor(hks, dtype=torch.long, device=kc.device)
        k = raw_numpy(kc.index_select(0, idx).index_select(2, hsel).cpu())
        v = raw_numpy(vc.index_select(0, idx).index_select(2, hsel).cpu())
        table = np.arange(n, dtype=np.int64)[None, :]
        ctx = np.array([c], dtype=np.int64)
        slot = oracle.paging.decode_slot_mapping(table, ctx, bs)
        hsel_cpu = torch.tensor(hks, dtype=torch.long)
        oracle.store.kv_store(raw_numpy(w.k_new[i:i + 1].cpu().index_select(1, hsel_cpu)),
                              raw_numpy(w.v_new[i:i + 1].cpu().index_select(1, hsel_cpu)), slot, k, v)
        kf = from_raw(k, dt).double().numpy()
        vf = from_raw(v, dt).double().numpy()
        q = w.q[i:i + 1, heads].double().cpu().numpy()
        res[i] = (heads, oracle.attention.decode_attention(q, kf, vf, table, ctx, w.scale)[0])
    return res


def partition_ctas_per_row(context_lens, grid, chunk=16):
    """How many partition CTAs share each row: the work is the flat list of
    (row, 16-token chunk) pairs cut into `grid` equal contiguous slices."""
    n = -(-np.maximum(np.asarray(context_lens, dtype=np.int64), 0) // chunk)
    P = np.concatenate([[0], np.cumsum(n)[:-1]])
    C = int(n.sum())
    starts = np.array([(C * c) // grid for c in range(grid + 1)], dtype=np.int64)
    first = np.searchsorted(starts, P, side="right") - 1
    last = np.searchsorted(starts, P + np.maximum(n, 1) - 1, side="right") - 1
    return np.where(n > 0, last - first + 1, 0)
