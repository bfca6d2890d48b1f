"""Paged decode attention on the GPU against the float64 oracle.

Tolerances: max abs error <= 1e-4 for fp32 caches; for fp16/bf16,
||o - ref||_inf / max(||ref||_inf, 1e-6) <= 2e-2 per (row, head), fp32
accumulation in the kernel.  Every workload NaN-poisons cache rows outside
the contexts and table entries past a row's blocks are -1, so a kernel that
reads or weights them fails.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import configs
from gpu_helpers import (require_gpu, oracle_store_f64, check_attention, gather_rows_for_oracle,
                         oracle_sampled, oracle_rows_by_kv_head, partition_ctas_per_row)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def small_variants():
    return {
        "tiny": configs.TINY,
        "nanochat": configs.NANOCHAT,
        "qwen3_small": configs.QWEN3.scaled(num_seqs=6, ctx_args=(1, 700), pool_blocks=48, num_layers=3,
                                            vocab=2048),
        "grok1_small": configs.GROK1.scaled(num_seqs=3, ctx_args=(300,), vocab=2048),
        "grok1_ragged": configs.GROK1.scaled(num_seqs=5, ctx_kind="explicit", ctx_args=(1, 15, 16, 17, 250),
                                             table_kind="perm", vocab=2048),
        "longctx_small": configs.LONGCTX.scaled(num_seqs=6, ctx_args=(1, 3000), vocab=2048),
        # many short rows, some empty: whole rows finish inside one CTA and
        # empty rows must come out as zeros
        "short_rows": configs.GROK1.scaled(num_seqs=400, num_q_heads=16, num_kv_heads=8, ctx_kind="uniform",
                                           ctx_args=(0, 40), table_kind="perm", vocab=2048),
        "mqa_f16": configs.QWEN3.scaled(num_seqs=4, num_q_heads=8, num_kv_heads=1, head_dim=128,
                                        block_size=32, ctx_args=(1, 300), pool_blocks=0, num_layers=1,
                                        vocab=2048),
    }


def paths_for(cfg, pk):
    out = [pk.PATH_FMA]
    if cfg.dtype != "f32" and cfg.num_kv_heads in (8, 16):
        out.append(pk.PATH_MMA)
    return out


def run_attention(pk, w, path, cache=None, window=0):
    lay = w.layout
    if cache is None:
        cache = w.cache.to(DEV)
    kc, vc = cache[0, lay.layer], cache[1, lay.layer]
    tables = torch.from_numpy(lay.block_tables).to(DEV)
    ctx = torch.from_numpy(lay.context_lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = pk.slot_mapping(tables, ctx, w.cfg.block_size, lay.num_blocks, err=err)
    q = w.q.to(DEV)
    pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, kc, vc, err=err)
    out = pk.paged_decode_attention(q, kc, vc, tables, ctx, lay.max_context_len, w.scale, err=err, path=path,
                                    window=window)
    torch.cuda.synchronize()
    return out, err.item()


@pytest.mark.parametrize("name", list(small_variants()))
def test_attention_matches_oracle(name):
    pk = require_gpu()
    cfg = small_variants()[name]
    w = workloads.make_workload(cfg)
    kf, vf, _ = oracle_store_f64(w)
    lay = w.layout
    ref = oracle.attention.decode_attention(w.q.double().numpy(), kf, vf, lay.block_tables,
                                            lay.context_lens, w.scale)
    for path in paths_for(cfg, pk):
        out, err = run_attention(pk, w, path)
        assert err == 0
        check_attention(out.double().cpu().numpy(), ref, w.q.dtype)
        zero_rows = np.nonzero(lay.context_lens == 0)[0]
        if len(zero_rows):
            assert torch.all(out[torch.from_numpy(zero_rows).to(DEV)] == 0)


def test_single_token_context_returns_v_exactly():
    pk = require_gpu()
    cfg = configs.GROK1.scaled(num_seqs=4, ctx_kind="explicit", ctx_args=(1, 1, 1, 1), table_kind="perm")
    w = workloads.make_workload(cfg)
    for path in paths_for(cfg, pk):
        out, err = run_attention(pk, w, path)
        assert err == 0
        G = cfg.group
        for i in range(4):
            for h in range(cfg.num_q_heads):
                assert torch.equal(out[i, h].cpu(), w.v_new[i, h // G])


def test_bad_block_id_is_flagged_not_read():
    pk = require_gpu()
    cfg = configs.GROK1.scaled(num_seqs=2, ctx_args=(64,), vocab=2048)
    w = workloads.make_workload(cfg)
    lay = w.layout
    lay.block_tables[1, 2] = lay.num_blocks + 5           # outside the pool
    cache = w.cache.to(DEV)
    tables = torch.from_numpy(lay.block_tables).to(DEV)
    ctx = torch.from_numpy(lay.context_lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk.paged_decode_attention(w.q.to(DEV), cache[0, 0], cache[1, 0], tables, ctx, lay.max_context_len,
                              w.scale, err=err)
    torch.cuda.synchronize()
    assert err.item() & pk.ERR_BLOCK_ID


@pytest.mark.parametrize("name", ["grok1", "qwen3", "longctx"])
def test_full_size_sampled_rows(name):
    """The benchmark's shapes and launch configuration, checked on sampled
    (row, head) pairs against the oracle, plus FMA/MMA agreement on every
    output element."""
    pk = require_gpu()
    cfg = configs.CONFIGS[name]
    w = workloads.make_workload(cfg, device=DEV)
    lay = w.layout
    rng = np.random.default_rng(0)
    longest = int(np.argmax(lay.context_lens))
    rows = sorted(set([0, longest, lay.num_seqs - 1] + rng.choice(lay.num_seqs, 3, replace=False).tolist()))
    heads = sorted(set([0, cfg.num_q_heads - 1] + rng.choice(cfg.num_q_heads, 2, replace=False).tolist()))
    gathered = gather_rows_for_oracle(w, rows)            # before any kernel touches the cache
    ref, pairs = oracle_sampled(w, gathered, rows, heads)
    outs = {}
    for path in paths_for(cfg, pk):
        out, err = run_attention(pk, w, path, cache=w.cache)
        assert err == 0
        o = out[torch.tensor(rows, device=DEV)].double().cpu().numpy()
        check_attention(o, ref, w.q.dtype, pairs=pairs)
        assert torch.isfinite(out).all()
        outs[path] = out.float()
    if len(outs) == 2:
        a, b = outs[pk.PATH_FMA], outs[pk.PATH_MMA]
        rel = (a - b).abs().amax(dim=-1) / a.abs().amax(dim=-1).clamp_min(1e-6)
        assert float(rel.max()) <= 2 * 2e-2


@pytest.mark.parametrize("name", ["grok1", "qwen3", "longctx"])
def test_full_size_every_row_against_oracle(name):
    """The benchmark's shapes and launch configuration, every row against the
    oracle: grok1 and qwen3 with every head, longctx with one KV head per row
    (rotating over the heads) and its whole query group.  The stream-K slices
    cut many rows across three or more CTAs (the merge of several partial
    records); the test asserts that such rows exist and are among those
    checked."""
    pk = require_gpu()
    cfg = configs.CONFIGS[name]
    w = workloads.make_workload(cfg, device=DEV)
    lay = w.layout
    B, Hkv = lay.num_seqs, cfg.num_kv_heads
    if name == "longctx":
        kv_heads = {i: [i % Hkv] for i in range(B)}
    else:
        kv_heads = {i: list(range(Hkv)) for i in range(B)}
    ref = oracle_rows_by_kv_head(w, range(B), kv_heads)      # before any kernel touches the cache
    ws = pk.decode_workspace_bytes(B, cfg.num_q_heads, cfg.head_dim, lay.max_context_len)
    grid = ws // (2 * cfg.num_q_heads * (cfg.head_dim + 4) * 4)
    spans = partition_ctas_per_row(lay.context_lens, grid)
    assert spans.max() >= 3, spans.max()
    for path in paths_for(cfg, pk):
        out, err = run_attention(pk, w, path, cache=w.cache)
        assert err == 0
        o = out.double().cpu().numpy()
        for i in range(B):
            heads, r = ref[i]
            check_attention(o[i:i + 1, heads], r[None], w.q.dtype)


def test_workspace_is_reusable_without_clearing():
    """One workspace, never cleared, serves repeated calls unchanged."""
    pk = require_gpu()
    cfg = configs.GROK1.scaled(num_seqs=7, ctx_kind="explicit", ctx_args=(700, 1, 0, 333, 2048, 17, 1500),
                               table_kind="perm", vocab=2048)
    w = workloads.make_workload(cfg)
    lay = w.layout
    cache = w.cache.to(DEV)
    tables = torch.from_numpy(lay.block_tables).to(DEV)
    ctx = torch.from_numpy(lay.context_lens).to(DEV)
    slots = pk.slot_mapping(tables, ctx, cfg.block_size, lay.num_blocks)
    pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, cache[0, 0], cache[1, 0])
    nbytes = pk.decode_workspace_bytes(lay.num_seqs, cfg.num_q_heads, cfg.head_dim, lay.max_context_len)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=DEV)      # garbage on purpose
    outs = [pk.paged_decode_attention(w.q.to(DEV), cache[0, 0], cache[1, 0], tables, ctx, lay.max_context_len,
                                      w.scale, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.isfinite(outs[0]).all()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert torch.all(outs[0][2] == 0)                     # the empty row


@pytest.mark.parametrize("name", ["qwen3_small", "grok1_ragged", "longctx_small", "short_rows", "mqa_f16", "tiny"])
@pytest.mark.parametrize("window", [1, 17, 256, 1000])
def test_sliding_window_matches_oracle(name, window):
    """Newest `window` positions only; cache rows before the window hold NaN
    in the poisoned workloads only past the context, so the window start
    must be exact for the result to match."""
    pk = require_gpu()
    cfg = small_variants()[name]
    w = workloads.make_workload(cfg)
    kf, vf, _ = oracle_store_f64(w)
    lay = w.layout
    ref = oracle.attention.decode_attention(w.q.double().numpy(), kf, vf, lay.block_tables,
                                            lay.context_lens, w.scale, window=window)
    for path in paths_for(cfg, pk):
        out, err = run_attention(pk, w, path, window=window)
        assert err == 0
        check_attention(out.double().cpu().numpy(), ref, w.q.dtype)


def test_sliding_window_never_reads_before_the_window():
    """Rows before each row's window are overwritten with NaN after the store:
    the windowed output stays finite and equal to the clean run."""
    pk = require_gpu()
    cfg = configs.GROK1.scaled(num_seqs=4, ctx_kind="explicit", ctx_args=(300, 40, 1, 129), table_kind="perm",
                               vocab=2048)
    w = workloads.make_workload(cfg)
    lay = w.layout
    W = 33
    cache = w.cache.to(DEV)
    clean, err = run_attention(pk, w, pk.PATH_AUTO, cache=cache, window=W)
    assert err == 0
    bs = cfg.block_size
    for i in range(lay.num_seqs):
        c = int(lay.context_lens[i])
        for j in range(max(0, c - W)):
            blk = int(lay.block_tables[i, j // bs])
            cache[:, lay.layer, blk, j % bs] = float("nan")
    dirty, err = run_attention(pk, w, pk.PATH_AUTO, cache=cache, window=W)
    assert err == 0
    assert torch.isfinite(dirty).all() and torch.equal(dirty, clean)


@pytest.mark.parametrize("name", ["qwen3", "longctx"])
def test_sliding_window_full_size_sampled_rows(name):
    pk = require_gpu()
    cfg = configs.CONFIGS[name]
    w = workloads.make_workload(cfg, device=DEV)
    lay = w.layout
    W = 1024
    rng = np.random.default_rng(1)
    longest = int(np.argmax(lay.context_lens))
    rows = sorted(set([0, longest, lay.num_seqs - 1] + rng.choice(lay.num_seqs, 3, replace=False).tolist()))
    heads = sorted(set([0, cfg.num_q_heads - 1] + rng.choice(cfg.num_q_heads, 2, replace=False).tolist()))
    gathered = gather_rows_for_oracle(w, rows)
    ref, pairs = oracle_sampled(w, gathered, rows, heads, window=W)
    for path in paths_for(cfg, pk):
        out, err = run_attention(pk, w, path, cache=w.cache, window=W)
        assert err == 0
        o = out[torch.tensor(rows, device=DEV)].double().cpu().numpy()
        check_attention(o, ref, w.q.dtype, pairs=pairs)


# ---------------------------------------------------------------- shared prefix
def prefix_variants():
    """Batches whose rows share their first `prefix` cached tokens (the same
    physical blocks at the start of every table), with the prefix length."""
    nano = configs.NANOCHAT
    return {
        "nanochat": (nano, 1024),
        "g6_head128": (nano.scaled(num_q_heads=48, num_kv_heads=8, ctx_args=(512, 200)), 512),
        "g8_rows12": (nano.scaled(num_seqs=12, num_q_heads=64, num_kv_heads=8, ctx_args=(256, 300)), 256),
        "g2_head64_f16": (nano.scaled(num_q_heads=16, num_kv_heads=8, head_dim=64, dtype="f16",
                                      ctx_args=(160, 40)), 160),
        "one_block_prefix": (nano.scaled(num_seqs=5, ctx_args=(16, 70)), 16),
        "block32": (nano.scaled(num_seqs=7, block_size=32, ctx_args=(320, 90)), 320),
        "many_rows": (nano.scaled(num_seqs=64, ctx_args=(128, 20)), 128),
    }


def run_prefix_attention(pk, w, prefix, workspace_fill=None):
    lay = w.layout
    cache = w.cache.to(DEV)
    kc, vc = cache[0, lay.layer], cache[1, lay.layer]
    tables = torch.from_numpy(lay.block_tables).to(DEV)
    ctx = torch.from_numpy(lay.context_lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = pk.slot_mapping(tables, ctx, w.cfg.block_size, lay.num_blocks, err=err)
    pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, kc, vc, err=err)
    ws = None
    if workspace_fill is not None:
        n = pk.decode_prefix_workspace_bytes(lay.num_seqs, w.cfg.num_q_heads, w.cfg.num_kv_heads, w.cfg.head_dim,
                                             lay.max_context_len, prefix)
        ws = torch.full((n,), workspace_fill, dtype=torch.uint8, device=DEV)
    out = pk.paged_decode_attention_prefix(w.q.to(DEV), kc, vc, tables, ctx, lay.max_context_len, w.scale, prefix,
                                           workspace=ws, err=err)
    torch.cuda.synchronize()
    return out, err.item()


@pytest.mark.parametrize("name", list(prefix_variants()))
def test_shared_prefix_attention_matches_oracle(name):
    """Every row against the oracle's plain attention over its own table (the
    prefix blocks are shared in the tables, so both read the same rows)."""
    pk = require_gpu()
    cfg, prefix = prefix_variants()[name]
    w = workloads.make_workload(cfg)
    lay = w.layout
    nb = prefix // cfg.block_size
    assert (lay.block_tables[:, :nb] == lay.block_tables[0, :nb]).all()
    assert (lay.context_lens > prefix).all()
    kf, vf, _ = oracle_store_f64(w)
    ref = oracle.attention.decode_attention(w.q.double().numpy(), kf, vf, lay.block_tables, lay.context_lens, w.scale)
    out, err = run_prefix_attention(pk, w, prefix, workspace_fill=0x7F)      # the workspace needs no clearing
    assert err == 0
    check_attention(out.double().cpu().numpy(), ref, w.q.dtype)
    again, _ = run_prefix_attention(pk, w, prefix)
    assert torch.equal(out, again)


@pytest.mark.parametrize("name,prefix", [("tiny", 16), ("qwen3_small", 256), ("nanochat", 0)])
def test_shared_prefix_call_falls_back_to_the_plain_kernel(name, prefix):
    """fp32 caches, 16 KV heads, or no prefix: the same result as the plain call."""
    pk = require_gpu()
    cfg = small_variants()[name]
    w = workloads.make_workload(cfg)
    lay = w.layout
    plain, err = run_attention(pk, w, pk.PATH_AUTO)
    assert err == 0
    pre, err = run_prefix_attention(pk, w, prefix)
    assert err == 0
    assert torch.equal(plain, pre)


def test_shared_prefix_rejects_partial_blocks_and_flags_short_rows():
    pk = require_gpu()
    cfg, prefix = prefix_variants()["one_block_prefix"]
    w = workloads.make_workload(cfg)
    with pytest.raises(pk.PkvdError):
        run_prefix_attention(pk, w, 8)                       # not a whole block
    # a row whose context does not reach past the prefix is flagged
    lay = w.layout
    lay.context_lens[2] = prefix
    _, err = run_prefix_attention(pk, w, prefix)
    assert err & pk.ERR_CONTEXT
