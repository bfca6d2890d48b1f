"""The five seeded synthetic decode workloads, as plain data.

Each workload is one decode step of a paged-KV engine: every sequence holds
``context_len - 1`` cached tokens plus the token being decoded now (whose K/V
is stored this step), and a row of vocabulary logits to sample from.

Shapes follow the engines the pages walk through:

* tiny: a hand-sized case the oracle finishes instantly.
* qwen3: nano-vllm's Qwen3-0.6B sizing ("Model Runner", section "allocated kv
  cache": 28 layers, block 256, 16 KV heads of 64, fp16).
* nanochat: one prefill shared by N samples ("04 · Engine", sections 2-3:
  prefill once, clone the cache N ways).
* grok1: Grok-1's static padded batch (48 query / 8 KV heads of 128, bf16;
  "第 8 章 runners.py 推理引擎", section 8.5 KV cache shapes).
* longctx: a long-context fragmented stress case.

Nothing here computes any part of the decode method; this module only names
sizes and distributions.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    index: int                     # 1..5, master seed is 1000 + index
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                     # "f32" | "f16" | "bf16" for q, K/V cache, out
    ctx_kind: str                  # how context lengths are drawn (see synth.py)
    ctx_args: tuple
    table_kind: str                # "perm" | "contiguous" | "shared_prefix"
    num_layers: int = 1            # layers held by the cache tensor
    pool_blocks: int = 0           # 0 = exactly the blocks the sequences need
    vocab: int = 1000
    logits_dtype: str = "f32"
    logits_std: float = 2.0
    temperature: tuple = ("const", 1.0)   # ("const", T) | ("uniform", lo, hi)
    top_k: int = 0
    top_p: float = 1.0
    kv_std: float = 1.0
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def itemsize(self) -> int:
        return {"f32": 4, "f16": 2, "bf16": 2}[self.dtype]

    @property
    def logits_itemsize(self) -> int:
        return {"f32": 4, "f16": 2, "bf16": 2}[self.logits_dtype]

    def scaled(self, **kw) -> "DecodeConfig":
        """A smaller variant with the same head/block/dtype structure."""
        return replace(self, **kw)


TINY = DecodeConfig(
    name="tiny", index=1, num_seqs=4, num_q_heads=4, num_kv_heads=2,
    head_dim=64, block_size=16, dtype="f32",
    ctx_kind="fixed", ctx_args=(1, 17, 33, 50),
    table_kind="perm", pool_blocks=32,
    vocab=1000, logits_dtype="f32", logits_std=2.0,
    temperature=("const", 1.0), top_k=0, top_p=1.0,
    description="tiny paged decode: 4 seqs, ctx {1,17,33,50}, 4 q / 2 kv heads, "
                "head_dim 64, block 16, 32-block pool, f32; logits [4,1000] f32 "
                "N(0,2), T=1 (and T=0 greedy in tests)",
)

QWEN3 = DecodeConfig(
    name="qwen3", index=2, num_seqs=64, num_q_heads=16, num_kv_heads=16,
    head_dim=64, block_size=256, dtype="f16",
    ctx_kind="uniform", ctx_args=(128, 4096),
    table_kind="perm", num_layers=28, pool_blocks=1024,
    vocab=151936, logits_dtype="f16", logits_std=3.0,
    temperature=("uniform", 0.6, 1.0), top_k=0, top_p=0.95,
    description="Qwen3-0.6B-shaped decode step: batch 64, 16 q / 16 kv heads, "
                "head_dim 64, block 256, fp16 cache [2,28,1024,256,16,64] "
                "(one layer per call), ctx U[128,4096], shuffled tables; "
                "fp16 logits [64,151936] N(0,3), T U[0.6,1.0], top_p 0.95",
)

NANOCHAT = DecodeConfig(
    name="nanochat", index=3, num_seqs=16, num_q_heads=8, num_kv_heads=8,
    head_dim=128, block_size=16, dtype="bf16",
    ctx_kind="shared_prefix", ctx_args=(1024, 255),
    table_kind="shared_prefix",
    vocab=65536, logits_dtype="bf16", logits_std=2.0,
    temperature=("const", 1.0), top_k=50, top_p=1.0,
    description="nanochat one-prefill-N-samples: 16 rows sharing a 1024-token "
                "prefix (same physical blocks) + 0-255 private tokens, "
                "8 q / 8 kv heads, head_dim 128, block 16, bf16; bf16 logits "
                "[16,65536] N(0,2), T=1, top_k 50",
)

GROK1 = DecodeConfig(
    name="grok1", index=4, num_seqs=32, num_q_heads=48, num_kv_heads=8,
    head_dim=128, block_size=16, dtype="bf16",
    ctx_kind="fixed_all", ctx_args=(2048,),
    table_kind="contiguous",
    vocab=131072, logits_dtype="bf16", logits_std=2.0,
    temperature=("const", 0.01), top_k=0, top_p=1.0,
    description="Grok-1-shaped static batch: 32 seqs padded to 2048, 48 q / 8 kv "
                "heads (group 6), head_dim 128, block 16, bf16, contiguous "
                "tables; bf16 logits [32,131072] N(0,2), T=0.01, top_p 1.0",
)

LONGCTX = DecodeConfig(
    name="longctx", index=5, num_seqs=256, num_q_heads=64, num_kv_heads=8,
    head_dim=128, block_size=16, dtype="bf16",
    ctx_kind="loguniform", ctx_args=(512, 32768),
    table_kind="perm",
    vocab=128256, logits_dtype="bf16", logits_std=2.0,
    temperature=("const", 0.8), top_k=0, top_p=0.9,
    description="long-context fragmented stress: 256 seqs, ctx log-uniform "
                "[512,32768], 64 q / 8 kv heads, head_dim 128, block 16, bf16, "
                "tables from a random permutation of the pool; bf16 logits "
                "[256,128256] N(0,2), T=0.8, top_p 0.9, per-row Philox seeds",
)

CONFIGS = {c.name: c for c in (TINY, QWEN3, NANOCHAT, GROK1, LONGCTX)}
BY_INDEX = {c.index: c for c in CONFIGS.values()}


def get(name_or_index) -> DecodeConfig:
    if isinstance(name_or_index, int) or str(name_or_index).isdigit():
        return BY_INDEX[int(name_or_index)]
    return CONFIGS[name_or_index]
