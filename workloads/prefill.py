"""Seeded synthetic varlen prefill batches (inputs only, no prefill arithmetic).

A batch is what a paged engine schedules for one prefill step (nano-vllm
"Model Runner" notes, sections "prepare Prefill" and "prefix cache"): per
sequence a number of new tokens and a number of already cached tokens (a
prefix-cache hit, or the earlier chunks of a chunked prefill), block tables
filled by the scheduler before the step, the new tokens' q / k / v rows and a
one-layer paged cache holding the cached prefixes.

Recipe (master seed ``2000 + config.index``, ``numpy.random.Generator``):

* stream ``[seed, 0]``: new-token counts, cached block counts, then the
  physical-block permutation;
* stream ``[seed, 1]``: q, new K, new V, then the cache, float32 normal
  draws rounded to the storage dtype (round to nearest even).

Cached prefixes are whole blocks.  With ``prefix_kind="shared"`` every
sequence's cached blocks are a leading run of one common list of physical
blocks (a system prompt cached once and hit by all); with ``"private"`` each
sequence owns its cached blocks (earlier chunks of its own prompt).  Cache
rows that no sequence holds before the store (the new tokens' rows, the tail
of each last block, blocks no table names) are NaN, so a kernel that reads a
row outside a context, or before the store, poisons its output.  Table
entries past a sequence's last block are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    index: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    q_kind: str                  # "fixed" (q_args = per-seq counts), "const", "uniform"
    q_args: tuple
    hit_kind: str                # "fixed" (per-seq cached blocks), "uniform" (0..hit_args[0]), "chunks"
    hit_args: tuple
    prefix_kind: str = "private"  # "shared" or "private"
    extra_blocks: int = 4
    window: int = 0
    description: str = ""

    @property
    def seed(self) -> int:
        return 2000 + self.index

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "PrefillConfig":
        return replace(self, **kw)


PF_TINY = PrefillConfig(
    name="prefill_tiny", index=1, num_seqs=5, num_q_heads=4, num_kv_heads=2, head_dim=64,
    block_size=16, dtype="f16", q_kind="fixed", q_args=(1, 17, 0, 130, 64),
    hit_kind="fixed", hit_args=(0, 2, 1, 3, 0), prefix_kind="private",
    description="5 seqs with 1/17/0/130/64 new tokens after 0/2/1/3/0 cached blocks of 16, "
                "4 q / 2 kv heads of 64, f16")

QWEN3_PREFILL = PrefillConfig(
    name="qwen3_prefill", index=2, num_seqs=16, num_q_heads=16, num_kv_heads=16, head_dim=64,
    block_size=256, dtype="f16", q_kind="uniform", q_args=(256, 2048),
    hit_kind="uniform", hit_args=(3,), prefix_kind="shared",
    description="Qwen3-0.6B-shaped prefill batch: 16 prompts of U[256,2048] new tokens, "
                "0-3 blocks of a shared 768-token system prompt cached (prefix-cache hits), "
                "16 q / 16 kv heads of 64, block 256, f16")

GROK1_PREFILL = PrefillConfig(
    name="grok1_prefill", index=3, num_seqs=8, num_q_heads=48, num_kv_heads=8, head_dim=128,
    block_size=16, dtype="bf16", q_kind="const", q_args=(1024,),
    hit_kind="fixed", hit_args=(0,) * 8, prefix_kind="private",
    description="Grok-1-shaped prefill: 8 prompts padded to the 1024-token bucket, nothing "
                "cached, 48 q / 8 kv heads of 128, block 16, bf16")

CHUNKED_PREFILL = PrefillConfig(
    name="chunked_prefill", index=4, num_seqs=4, num_q_heads=64, num_kv_heads=8, head_dim=128,
    block_size=16, dtype="bf16", q_kind="const", q_args=(2048,),
    hit_kind="chunks", hit_args=(2048, 7), prefix_kind="private",
    description="chunked prefill of long prompts: 4 seqs, a 2048-token chunk each after "
                "0-7 earlier chunks of 2048 (cached), 64 q / 8 kv heads of 128, block 16, bf16")

PREFILL_CONFIGS = {c.name: c for c in (PF_TINY, QWEN3_PREFILL, GROK1_PREFILL, CHUNKED_PREFILL)}


@dataclass
class PrefillBatch:
    cfg: PrefillConfig
    cu_seqlens_q: np.ndarray    # int32 [B + 1]
    cu_seqlens_k: np.ndarray    # int32 [B + 1]
    block_tables: np.ndarray    # int32 [B, max_blocks]; -1 = unused
    num_blocks: int
    q: torch.Tensor             # [total_q, Hq, D]
    k_new: torch.Tensor         # [total_q, Hkv, D]
    v_new: torch.Tensor         # [total_q, Hkv, D]
    cache: torch.Tensor         # [2, num_blocks, bs, Hkv, D]; NaN where nothing is held yet

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)

    @property
    def k_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_k)

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max()) if len(self.q_lens) else 0

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.cfg.head_dim)


def _counts(cfg: PrefillConfig, rng: np.random.Generator):
    B = cfg.num_seqs
    if cfg.q_kind == "fixed":
        q = np.array(cfg.q_args, dtype=np.int64)
    elif cfg.q_kind == "const":
        q = np.full(B, cfg.q_args[0], dtype=np.int64)
    elif cfg.q_kind == "uniform":
        q = rng.integers(cfg.q_args[0], cfg.q_args[1] + 1, size=B)
    else:
        raise ValueError(cfg.q_kind)
    bs = cfg.block_size
    if cfg.hit_kind == "fixed":
        hit_blocks = np.array(cfg.hit_args, dtype=np.int64)
    elif cfg.hit_kind == "uniform":
        hit_blocks = rng.integers(0, cfg.hit_args[0] + 1, size=B)
    elif cfg.hit_kind == "chunks":
        chunk, most = cfg.hit_args
        assert chunk % bs == 0
        hit_blocks = rng.integers(0, most + 1, size=B) * (chunk // bs)
    else:
        raise ValueError(cfg.hit_kind)
    return q, hit_blocks


def make_prefill_batch(cfg: PrefillConfig, seed: int | None = None) -> PrefillBatch:
    """Draw one prefill step's inputs on the host (numpy PCG64)."""
    seed = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    B, bs = cfg.num_seqs, cfg.block_size
    q_lens, hit_blocks = _counts(cfg, rng)
    cached = hit_blocks * bs
    k_lens = q_lens + cached
    nblk = [-(-int(k) // bs) for k in k_lens]
    width = max(1, max(nblk) if nblk else 1)

    shared = int(hit_blocks.max()) if (cfg.prefix_kind == "shared" and B) else 0
    private = [n - (int(h) if cfg.prefix_kind == "shared" else 0) for n, h in zip(nblk, hit_blocks)]
    pool = shared + int(sum(private)) + cfg.extra_blocks
    perm = rng.permutation(pool).astype(np.int32)
    tables = np.full((B, width), -1, dtype=np.int32)
    at = shared
    for i in range(B):
        h = int(hit_blocks[i]) if cfg.prefix_kind == "shared" else 0
        tables[i, :h] = perm[:h]
        tables[i, h:h + private[i]] = perm[at:at + private[i]]
        at += private[i]

    vrng = np.random.Generator(np.random.PCG64([seed, 1]))
    dt = TORCH_DTYPES[cfg.dtype]
    T = int(q_lens.sum())
    Hq, Hkv, D = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    q = torch.from_numpy(vrng.standard_normal((T, Hq, D), dtype=np.float32)).to(dt)
    k_new = torch.from_numpy(vrng.standard_normal((T, Hkv, D), dtype=np.float32)).to(dt)
    v_new = torch.from_numpy(vrng.standard_normal((T, Hkv, D), dtype=np.float32)).to(dt)
    cache = torch.from_numpy(vrng.standard_normal((2, pool, bs, Hkv, D), dtype=np.float32)).to(dt)

    # rows held before the store: the cached prefix of every sequence
    held = np.zeros((pool, bs), dtype=bool)
    for i in range(B):
        for j in range(int(hit_blocks[i])):
            held[tables[i, j], :] = True
    cache[:, torch.from_numpy(~held)] = float("nan")

    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    return PrefillBatch(cfg, cu_q, cu_k, tables, int(pool), q, k_new, v_new, cache)
