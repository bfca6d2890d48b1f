"""Varlen paged prefill on the GPU against the float64 oracle.

Store: the cache after pkvd_kv_store_prefill and its slot mapping must equal,
bit for bit, the oracle's slot mapping and store on the same host inputs.
Attention: per (token, head) ||o - ref||_inf / max(||ref||_inf, 1e-6) <= 2e-2
(16-bit K/V, fp32 accumulation, softmax weights rounded to the K/V type
for the second product).  Every batch NaN-poisons the cache rows nobody
holds before the store, so reading a row outside a context, or the new rows
before they are stored, fails.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import prefill as wp
from gpu_helpers import require_gpu, raw_numpy, from_raw, RTOL_16, ATOL_F32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def small_batches():
    return {
        "tiny": wp.PF_TINY,
        "qwen3_small": wp.QWEN3_PREFILL.scaled(num_seqs=4, q_args=(1, 300), extra_blocks=2),
        "grok1_small": wp.GROK1_PREFILL.scaled(num_seqs=2, q_args=(150,), hit_args=(0, 0)),
        "grok1_hits": wp.GROK1_PREFILL.scaled(num_seqs=3, q_kind="fixed", q_args=(70, 1, 129),
                                              hit_kind="fixed", hit_args=(5, 9, 0), prefix_kind="shared"),
        "mqa_g8_bf16": wp.PrefillConfig(name="mqa", index=7, num_seqs=3, num_q_heads=8, num_kv_heads=1,
                                        head_dim=128, block_size=32, dtype="bf16", q_kind="fixed",
                                        q_args=(33, 64, 200), hit_kind="fixed", hit_args=(1, 0, 2)),
        "g16_f16": wp.PrefillConfig(name="g16", index=8, num_seqs=2, num_q_heads=32, num_kv_heads=2,
                                    head_dim=64, block_size=64, dtype="f16", q_kind="fixed",
                                    q_args=(20, 9), hit_kind="fixed", hit_args=(1, 0)),
        "chunked_small": wp.CHUNKED_PREFILL.scaled(num_seqs=2, q_args=(96,), hit_args=(256, 2)),
        # block 8: one TMA box per 8-row swizzle atom; block 128: one box per K/V tile
        "bs8_f16_d128": wp.PrefillConfig(name="bs8", index=10, num_seqs=3, num_q_heads=8, num_kv_heads=2,
                                         head_dim=128, block_size=8, dtype="f16", q_kind="fixed",
                                         q_args=(41, 300, 7), hit_kind="fixed", hit_args=(3, 0, 20)),
        "bs128_bf16_d64": wp.PrefillConfig(name="bs128", index=11, num_seqs=3, num_q_heads=4, num_kv_heads=2,
                                           head_dim=64, block_size=128, dtype="bf16", q_kind="fixed",
                                           q_args=(129, 500, 2), hit_kind="fixed", hit_args=(1, 2, 0)),
        # fp32 caches: the CUDA-core path only
        "f32_d64": wp.PrefillConfig(name="f32a", index=12, num_seqs=3, num_q_heads=4, num_kv_heads=2, head_dim=64,
                                    block_size=16, dtype="f32", q_kind="fixed", q_args=(17, 40, 1),
                                    hit_kind="fixed", hit_args=(1, 0, 3)),
        "f32_d128_g4": wp.PrefillConfig(name="f32b", index=13, num_seqs=2, num_q_heads=8, num_kv_heads=2,
                                        head_dim=128, block_size=32, dtype="f32", q_kind="fixed", q_args=(70, 33),
                                        hit_kind="fixed", hit_args=(2, 0), prefix_kind="shared"),
    }


def oracle_cache(b):
    """The oracle's slot mapping and store on the host batch; returns float64
    K, V caches ([num_blocks, bs, Hkv, D]) and the slots."""
    slots = oracle.prefill.prefill_slot_mapping(b.block_tables, b.cu_seqlens_q, b.cu_seqlens_k,
                                                b.cfg.block_size)
    k = raw_numpy(b.cache[0])
    v = raw_numpy(b.cache[1])
    oracle.store.kv_store(raw_numpy(b.k_new), raw_numpy(b.v_new), slots, k, v)
    return k, v, slots


def to_f64(raw, dtype):
    return from_raw(raw, dtype).double().numpy()


def run_prefill(pk, b, window=0, max_seqlen_q=None, total_rows=None, path=None):
    cache = b.cache.to(DEV)
    kc, vc = cache[0], cache[1]
    tables = torch.from_numpy(b.block_tables).to(DEV)
    cu_q = torch.from_numpy(b.cu_seqlens_q).to(DEV)
    cu_k = torch.from_numpy(b.cu_seqlens_k).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    T = b.total_q if total_rows is None else total_rows
    q = torch.zeros((T,) + tuple(b.q.shape[1:]), dtype=b.q.dtype)
    k = torch.zeros((T,) + tuple(b.k_new.shape[1:]), dtype=b.k_new.dtype)
    v = torch.zeros_like(k)
    q[:b.total_q], k[:b.total_q], v[:b.total_q] = b.q, b.k_new, b.v_new
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    slots = torch.full((T,), -7, dtype=torch.int64, device=DEV)
    pk.kv_store_prefill(k, v, tables, cu_q, cu_k, kc, vc, slot_mapping=slots, err=err)
    out = torch.full_like(q, 1024.0)
    pk.prefill_attention(q, kc, vc, tables, cu_q, cu_k,
                         b.max_seqlen_q if max_seqlen_q is None else max_seqlen_q,
                         b.scale, window=window, out=out, err=err, path=pk.PATH_AUTO if path is None else path)
    torch.cuda.synchronize()
    return cache.cpu(), slots.cpu().numpy(), out.cpu(), int(err.item())


def check_rows(out, ref, pairs, f32=False):
    """16-bit caches: relative error per (token, head) <= 2e-2; fp32: max abs
    error <= 1e-4 (the decode attention's tolerances)."""
    worst = 0.0
    for t, h in pairs:
        o, r = out[t, h], ref[t, h]
        assert np.all(np.isfinite(o)), (t, h)
        if f32:
            e = float(np.abs(o - r).max())
            assert e <= ATOL_F32, (t, h, e)
        else:
            e = float(np.abs(o - r).max() / max(np.abs(r).max(), 1e-6))
            assert e <= RTOL_16, (t, h, e)
        worst = max(worst, e)
    return worst


@pytest.mark.parametrize("name", list(small_batches()))
def test_prefill_store_bit_exact(name):
    pk = require_gpu()
    b = wp.make_prefill_batch(small_batches()[name])
    k_ref, v_ref, slots_ref = oracle_cache(b)
    cache, slots, _, err = run_prefill(pk, b)
    assert err == 0
    np.testing.assert_array_equal(slots, slots_ref)
    np.testing.assert_array_equal(raw_numpy(cache[0]), k_ref)
    np.testing.assert_array_equal(raw_numpy(cache[1]), v_ref)


@pytest.mark.parametrize("path", ["tc", "mma", "fma"])
@pytest.mark.parametrize("window", [0, 1, 50, 200])
@pytest.mark.parametrize("name", list(small_batches()))
def test_prefill_attention_matches_oracle(name, window, path):
    cfg = small_batches()[name]
    if cfg.dtype == "f32" and path != "fma":
        pytest.skip("the tensor-core paths take 16-bit caches")
    pk = require_gpu()
    b = wp.make_prefill_batch(cfg)
    k_ref, v_ref, _ = oracle_cache(b)
    dt = b.cache.dtype
    ref = oracle.prefill.prefill_attention(b.q.double().numpy(), to_f64(k_ref, dt), to_f64(v_ref, dt),
                                           b.block_tables, b.cu_seqlens_q, b.cu_seqlens_k, b.scale,
                                           window=window)
    _, _, out, err = run_prefill(pk, b, window=window,
                                 path={"tc": pk.PATH_TC, "mma": pk.PATH_MMA, "fma": pk.PATH_FMA}[path])
    assert err == 0
    T, Hq, _ = ref.shape
    check_rows(out.double().numpy(), ref, [(t, h) for t in range(T) for h in range(Hq)], f32=cfg.dtype == "f32")


def test_rows_past_the_batch_are_untouched():
    pk = require_gpu()
    b = wp.make_prefill_batch(wp.PF_TINY)
    _, slots, out, err = run_prefill(pk, b, total_rows=b.total_q + 9)
    assert err == 0
    assert (slots[b.total_q:] == -1).all()
    assert (out[b.total_q:].float() == 1024.0).all()


def test_short_max_seqlen_flags_context():
    pk = require_gpu()
    b = wp.make_prefill_batch(wp.PF_TINY)
    _, _, out, err = run_prefill(pk, b, max_seqlen_q=64)     # one sequence has 130 new tokens
    assert err == pk.ERR_CONTEXT
    # the grid covers the last ceil(64 / tile) * tile tokens of each sequence
    # (tile = 128 // group query tokens); those of the long one are still right
    tile = 128 // b.cfg.group
    covered = -(-64 // tile) * tile
    k_ref, v_ref, _ = oracle_cache(b)
    dt = b.cache.dtype
    t1 = int(b.cu_seqlens_q[4])
    pairs = [(t, h) for t in range(t1 - covered, t1) for h in range(4)]
    ref = oracle.prefill.prefill_attention(b.q.double().numpy(), to_f64(k_ref, dt), to_f64(v_ref, dt),
                                           b.block_tables, b.cu_seqlens_q, b.cu_seqlens_k, b.scale, pairs=pairs)
    check_rows(out.double().numpy(), ref, pairs)


def test_bad_lengths_and_blocks_flag_errors():
    pk = require_gpu()
    b = wp.make_prefill_batch(wp.PF_TINY)
    bad = wp.PrefillBatch(b.cfg, b.cu_seqlens_q, b.cu_seqlens_k.copy(), b.block_tables.copy(), b.num_blocks,
                          b.q, b.k_new, b.v_new, b.cache)
    bad.cu_seqlens_k[2:] -= 40      # sequence 1: 17 new tokens but k_len 17 + 32 - 40 < 17
    _, slots, _, err = run_prefill(pk, bad)
    assert err & pk.ERR_CONTEXT
    assert (slots[b.cu_seqlens_q[1]:b.cu_seqlens_q[2]] == -1).all()
    bad2 = wp.PrefillBatch(b.cfg, b.cu_seqlens_q, b.cu_seqlens_k, b.block_tables.copy(), b.num_blocks,
                           b.q, b.k_new, b.v_new, b.cache)
    bad2.block_tables[4, 0] = b.num_blocks + 5
    _, slots, out, err = run_prefill(pk, bad2)
    assert err == pk.ERR_BLOCK_ID
    assert (slots[b.cu_seqlens_q[4]:b.cu_seqlens_q[4] + 16] == -1).all()
    assert torch.isfinite(out[:b.total_q].float()).all()


def test_chunked_prefill_on_device_matches_one_shot_oracle():
    """Three chunks run as three store + attention calls on the device; every
    chunk's rows equal the oracle's one-shot prefill of the whole prompt."""
    pk = require_gpu()
    cfg = wp.PrefillConfig(name="chunks", index=9, num_seqs=1, num_q_heads=12, num_kv_heads=2, head_dim=128,
                           block_size=16, dtype="bf16", q_kind="fixed", q_args=(301,), hit_kind="fixed",
                           hit_args=(0,))
    b = wp.make_prefill_batch(cfg)
    k_ref, v_ref, _ = oracle_cache(b)
    dt = b.cache.dtype
    ref = oracle.prefill.prefill_attention(b.q.double().numpy(), to_f64(k_ref, dt), to_f64(v_ref, dt),
                                           b.block_tables, b.cu_seqlens_q, b.cu_seqlens_k, b.scale)
    cache = b.cache.to(DEV)
    tables = torch.from_numpy(b.block_tables).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs, done = [], 0
    for m in (100, 1, 200):
        cu_q = torch.tensor([0, m], dtype=torch.int32, device=DEV)
        cu_k = torch.tensor([0, done + m], dtype=torch.int32, device=DEV)
        sl = slice(done, done + m)
        pk.kv_store_prefill(b.k_new[sl].to(DEV), b.v_new[sl].to(DEV), tables, cu_q, cu_k, cache[0], cache[1],
                            err=err)
        outs.append(pk.prefill_attention(b.q[sl].to(DEV), cache[0], cache[1], tables, cu_q, cu_k, m, b.scale,
                                         err=err))
        done += m
    torch.cuda.synchronize()
    assert err.item() == 0
    out = torch.cat(outs).cpu().double().numpy()
    check_rows(out, ref, [(t, h) for t in range(301) for h in range(12)])


@pytest.mark.parametrize("name", ["qwen3_prefill", "grok1_prefill", "chunked_prefill"])
def test_full_size_prefill_sampled(name):
    """The benchmark's batches at full size, launched as the benchmark does:
    the store bit-exact everywhere, attention on sampled (token, head) pairs
    (the first and last token of every sequence and 48 random ones)."""
    pk = require_gpu()
    b = wp.make_prefill_batch(wp.PREFILL_CONFIGS[name])
    k_ref, v_ref, slots_ref = oracle_cache(b)
    cache, slots, out, err = run_prefill(pk, b)
    assert err == 0
    np.testing.assert_array_equal(slots, slots_ref)
    np.testing.assert_array_equal(raw_numpy(cache[0]), k_ref)
    np.testing.assert_array_equal(raw_numpy(cache[1]), v_ref)
    rng = np.random.default_rng(5)
    Hq = b.cfg.num_q_heads
    toks = set()
    for i in range(b.cfg.num_seqs):
        if b.q_lens[i]:
            toks.update([int(b.cu_seqlens_q[i]), int(b.cu_seqlens_q[i + 1]) - 1])
    toks.update(int(t) for t in rng.integers(0, b.total_q, 48))
    pairs = [(t, int(rng.integers(0, Hq))) for t in sorted(toks)]
    dt = b.cache.dtype
    ref = oracle.prefill.prefill_attention(b.q.double().numpy(), to_f64(k_ref, dt), to_f64(v_ref, dt),
                                           b.block_tables, b.cu_seqlens_q, b.cu_seqlens_k, b.scale, pairs=pairs)
    check_rows(out.double().numpy(), ref, pairs)
