"""Seeded synthetic inputs for the decode step.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It draws inputs only: context lengths, block tables (the
scheduler's bookkeeping), query / new-K/V / cache / logit values and the
sampling parameters.  It holds none of the decode method's arithmetic (no
slot computation, no attention, no sampling).

Recipe (master seed ``1000 + config.index``):

* Layout (always on the host, ``numpy.random.Generator(PCG64(seed))``):
  context lengths, then the block-table permutation, then per-row sampling
  parameters (temperatures, Philox seeds).
* Values: on the host the same generator continues with q, new K, new V,
  the cache and the logits as float32 normal draws, rounded to the storage
  dtype with round-to-nearest-even.  On a CUDA device, a
  ``torch.Generator`` seeded with the master seed fills the same tensors in
  the same order (used for the multi-GB configurations).
* Every cache row that is not part of a sequence's context (rows at or after
  the new token's position in the last block, and blocks no table
  references) is set to NaN, so a kernel that reads or weights such a row
  poisons its output.  The new token's own row is NaN before the store.
* Block-table entries past a sequence's last block are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from .configs import DecodeConfig

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Layout:
    context_lens: np.ndarray      # int32 [B]; includes the token decoded now
    block_tables: np.ndarray      # int32 [B, max_blocks_per_seq]; -1 = unused
    num_blocks: int               # physical blocks in the pool
    layer: int                    # which cache layer this step exercises
    max_context_len: int          # bound the caller passes to the kernel

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def _draw_context_lens(cfg: DecodeConfig, rng: np.random.Generator, B: int):
    kind, args = cfg.ctx_kind, cfg.ctx_args
    if kind == "fixed":
        ctx = np.array(args, dtype=np.int64)[:B]
        bound = int(max(args))
    elif kind == "fixed_all":
        ctx = np.full(B, args[0], dtype=np.int64)
        bound = int(args[0])
    elif kind == "uniform":
        lo, hi = args
        ctx = rng.integers(lo, hi + 1, size=B)
        bound = int(hi)
    elif kind == "loguniform":
        lo, hi = args
        ctx = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=B)))
        ctx = np.clip(ctx, lo, hi).astype(np.int64)
        bound = int(hi)
    elif kind == "shared_prefix":
        prefix, max_private = args
        private = rng.integers(0, max_private + 1, size=B)
        ctx = prefix + private + 1
        bound = int(prefix + max_private + 1)
    elif kind == "explicit":
        ctx = np.array(args, dtype=np.int64)
        bound = int(ctx.max()) if len(ctx) else 0
    else:
        raise ValueError(kind)
    return ctx.astype(np.int32), bound


def make_layout(cfg: DecodeConfig, seed: int | None = None) -> Layout:
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    B, bs = cfg.num_seqs, cfg.block_size
    ctx, bound = _draw_context_lens(cfg, rng, B)
    nblk = [(-(-int(c) // bs)) for c in ctx]            # blocks each row owns
    width = max(1, -(-bound // bs))
    tables = np.full((B, width), -1, dtype=np.int32)

    if cfg.table_kind == "contiguous":
        pool = max(width * B, cfg.pool_blocks)
        for i in range(B):
            tables[i, : nblk[i]] = np.arange(i * width, i * width + nblk[i])
    elif cfg.table_kind == "perm":
        need = int(sum(nblk))
        pool = max(need, cfg.pool_blocks)
        perm = rng.permutation(pool).astype(np.int32)
        pos = 0
        for i in range(B):
            tables[i, : nblk[i]] = perm[pos: pos + nblk[i]]
            pos += nblk[i]
    elif cfg.table_kind == "shared_prefix":
        prefix_tokens = cfg.ctx_args[0]
        assert prefix_tokens % bs == 0
        npre = prefix_tokens // bs
        priv = [n - npre for n in nblk]
        pool = npre + int(sum(priv))
        pool = max(pool, cfg.pool_blocks)
        perm = rng.permutation(pool).astype(np.int32)
        tables[:, :npre] = perm[:npre]
        pos = npre
        for i in range(B):
            tables[i, npre: npre + priv[i]] = perm[pos: pos + priv[i]]
            pos += priv[i]
    else:
        raise ValueError(cfg.table_kind)

    layer = int(rng.integers(0, cfg.num_layers)) if cfg.num_layers > 1 else 0
    return Layout(ctx, tables, int(pool), layer, int(bound))


def _sampling_params(cfg: DecodeConfig, rng: np.random.Generator, B: int):
    t = cfg.temperature
    if t[0] == "const":
        temp = np.full(B, t[1], dtype=np.float32)
    else:
        temp = rng.uniform(t[1], t[2], size=B).astype(np.float32)
    top_k = np.full(B, cfg.top_k, dtype=np.int32)
    top_p = np.full(B, cfg.top_p, dtype=np.float32)
    seeds = rng.integers(0, 2**63 - 1, size=B, dtype=np.int64).astype(np.uint64)
    offsets = np.zeros(B, dtype=np.uint64)
    return temp, top_k, top_p, seeds, offsets


@dataclass
class Workload:
    cfg: DecodeConfig
    layout: Layout
    q: torch.Tensor            # [B, Hq, D]
    k_new: torch.Tensor        # [B, Hkv, D]
    v_new: torch.Tensor        # [B, Hkv, D]
    cache: torch.Tensor        # [2, L, num_blocks, bs, Hkv, D]; K = [0, layer]
    logits: torch.Tensor       # [B, V]
    temperature: np.ndarray    # f32 [B]
    top_k: np.ndarray          # i32 [B]
    top_p: np.ndarray          # f32 [B]
    seeds: np.ndarray          # u64 [B]
    offsets: np.ndarray        # u64 [B]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.cfg.head_dim)

    def k_cache(self) -> torch.Tensor:
        return self.cache[0, self.layout.layer]

    def v_cache(self) -> torch.Tensor:
        return self.cache[1, self.layout.layer]


def poison_rows(layout: Layout, block_size: int):
    """(used-block mask, list of (block, row) pairs) that must hold NaN.

    A row is outside every context if it sits at or after the new token's
    position inside a sequence's last block; a block is unused if no table
    references it.
    """
    used = np.zeros(layout.num_blocks, dtype=bool)
    rows = []
    for i, c in enumerate(layout.context_lens):
        c = int(c)
        n = -(-c // block_size)
        blocks = layout.block_tables[i, :n]
        used[blocks] = True
        if n:
            last = int(blocks[-1])
            first_free = (c - 1) % block_size      # the new token's row, then the tail
            for r in range(first_free, block_size):
                rows.append((last, r))
    return used, rows


def _fill_normal(t: torch.Tensor, gen, std: float = 1.0):
    if t.device.type == "cpu":
        raise RuntimeError("use the numpy path on the host")
    t.normal_(0.0, std, generator=gen)


def make_workload(cfg: DecodeConfig, device: str = "cpu", seed: int | None = None,
                  layout: Layout | None = None) -> Workload:
    """Draw one decode step's inputs.  ``device='cpu'`` uses numpy PCG64;
    ``device='cuda'`` draws the big tensors with a seeded torch generator."""
    seed = cfg.seed if seed is None else seed
    layout = make_layout(cfg, seed) if layout is None else layout
    # sampling params draw from a second stream so the layout stays fixed
    prng = np.random.Generator(np.random.PCG64([seed, 1]))
    temp, top_k, top_p, seeds, offsets = _sampling_params(cfg, prng, layout.num_seqs)

    B, Hq, Hkv, D, bs = layout.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    dt = TORCH_DTYPES[cfg.dtype]
    ldt = TORCH_DTYPES[cfg.logits_dtype]
    cache_shape = (2, cfg.num_layers, layout.num_blocks, bs, Hkv, D)

    if device == "cpu":
        rng = np.random.Generator(np.random.PCG64([seed, 2]))
        q = torch.from_numpy(rng.standard_normal((B, Hq, D), dtype=np.float32)).to(dt)
        k_new = torch.from_numpy((cfg.kv_std * rng.standard_normal((B, Hkv, D), dtype=np.float32))).to(dt)
        v_new = torch.from_numpy((cfg.kv_std * rng.standard_normal((B, Hkv, D), dtype=np.float32))).to(dt)
        cache = torch.from_numpy(cfg.kv_std * rng.standard_normal(cache_shape, dtype=np.float32)).to(dt)
        logits = torch.from_numpy(cfg.logits_std * rng.standard_normal((B, cfg.vocab), dtype=np.float32)).to(ldt)
    else:
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        q = torch.empty((B, Hq, D), dtype=dt, device=device)
        _fill_normal(q, gen)
        k_new = torch.empty((B, Hkv, D), dtype=dt, device=device)
        _fill_normal(k_new, gen, cfg.kv_std)
        v_new = torch.empty((B, Hkv, D), dtype=dt, device=device)
        _fill_normal(v_new, gen, cfg.kv_std)
        cache = torch.empty(cache_shape, dtype=dt, device=device)
        for kv in range(2):
            for l in range(cfg.num_layers):
                _fill_normal(cache[kv, l], gen, cfg.kv_std)
        logits = torch.empty((B, cfg.vocab), dtype=ldt, device=device)
        _fill_normal(logits, gen, cfg.logits_std)

    used, rows = poison_rows(layout, bs)
    nan = float("nan")
    unused = torch.from_numpy(np.nonzero(~used)[0]).to(cache.device)
    if unused.numel():
        cache[:, :, unused] = nan
    if rows:
        rb = torch.tensor([r[0] for r in rows], device=cache.device)
        rr = torch.tensor([r[1] for r in rows], device=cache.device)
        cache[:, :, rb, rr] = nan

    return Workload(cfg, layout, q, k_new, v_new, cache, logits,
                    temp, top_k, top_p, seeds, offsets)


@dataclass
class SamplerInputs:
    cfg: DecodeConfig
    logits: torch.Tensor       # [B, V] in the config's logits dtype
    temperature: np.ndarray    # f32 [B]
    top_k: np.ndarray          # i32 [B]
    top_p: np.ndarray          # f32 [B]
    seeds: np.ndarray          # u64 [B]
    offsets: np.ndarray        # u64 [B]


def make_sampler_inputs(cfg: DecodeConfig, device: str = "cpu", seed: int | None = None,
                        num_rows: int | None = None) -> SamplerInputs:
    """Only the sampler's inputs (logits + per-row parameters) of a config.

    The per-row parameters come from the same stream as make_workload's; the
    logits from their own stream, so this does not draw the KV cache."""
    seed = cfg.seed if seed is None else seed
    B = cfg.num_seqs if num_rows is None else num_rows
    prng = np.random.Generator(np.random.PCG64([seed, 1]))
    temp, top_k, top_p, seeds, offsets = _sampling_params(cfg, prng, B)
    ldt = TORCH_DTYPES[cfg.logits_dtype]
    if device == "cpu":
        rng = np.random.Generator(np.random.PCG64([seed, 3]))
        logits = torch.from_numpy(cfg.logits_std * rng.standard_normal((B, cfg.vocab), dtype=np.float32)).to(ldt)
    else:
        gen = torch.Generator(device=device)
        gen.manual_seed(seed + 7919)
        logits = torch.empty((B, cfg.vocab), dtype=ldt, device=device)
        _fill_normal(logits, gen, cfg.logits_std)
    return SamplerInputs(cfg, logits, temp, top_k, top_p, seeds, offsets)
