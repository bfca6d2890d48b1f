"""Seeded random shapes against the float64 oracle: decode attention (both
consumer paths, with and without a sliding window), the shared-prefix call,
and the sampler over random vocabularies, dtypes and cut parameters.

The fixed cases elsewhere pin each branch on purpose; these sweep the
combinations (head counts and groups, head_dim, block size, empty and
one-token rows, tables that are permuted or contiguous, ties in the logits)
with the same tolerances and exemptions.  Every case is drawn from a seeded
generator, so a failure names a reproducible case.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import configs
from gpu_helpers import require_gpu, oracle_store_f64, check_attention, sampling_exempt

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _attention_case(rng, i):
    dtype = str(rng.choice(["bf16", "f16", "f32"], p=[0.45, 0.45, 0.1]))
    hkv = int(rng.choice([1, 2, 4, 8, 16], p=[0.1, 0.1, 0.1, 0.5, 0.2]))
    if dtype == "f32" and hkv == 16:
        hkv = 8
    G = int(rng.choice([1, 2, 3, 4, 6, 8]))
    D = int(rng.choice([64, 128]))
    if hkv * D * (4 if dtype == "f32" else 2) > 2048:   # a K/V token row must fit the staging (two stages)
        D = 64
    cmax = int(rng.choice([1, 16, 40, 300, 2000]))
    cfg = configs.GROK1.scaled(index=300 + i, num_seqs=int(rng.integers(1, 24)), num_q_heads=hkv * G,
                               num_kv_heads=hkv, head_dim=D,
                               block_size=int(rng.choice([16, 32, 64, 128, 256])), dtype=dtype,
                               ctx_kind="uniform", ctx_args=(0, cmax),
                               table_kind=str(rng.choice(["perm", "contiguous"])), vocab=1024)
    return cfg, int(rng.choice([0, 0, 1, 7, 16, 100]))


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_attention_shapes_match_oracle(seed):
    pk = require_gpu()
    rng = np.random.default_rng(5000 + seed)
    checked = 0
    for i in range(12):
        cfg, window = _attention_case(rng, seed * 100 + i)
        w = workloads.make_workload(cfg)
        lay = w.layout
        if lay.block_tables.shape[1] == 0 or int(lay.context_lens.max()) == 0:
            continue
        kf, vf, _ = oracle_store_f64(w)
        ref = oracle.attention.decode_attention(w.q.double().numpy(), kf, vf, lay.block_tables, lay.context_lens,
                                                w.scale, window=window)
        cache = w.cache.to(DEV)
        kc, vc = cache[0, lay.layer], cache[1, lay.layer]
        tables = torch.from_numpy(lay.block_tables).to(DEV)
        ctx = torch.from_numpy(lay.context_lens).to(DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        slots = pk.slot_mapping(tables, ctx, cfg.block_size, lay.num_blocks, err=err)
        pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, kc, vc, err=err)
        paths = [pk.PATH_FMA] + ([pk.PATH_MMA] if cfg.dtype != "f32" and cfg.num_kv_heads in (8, 16) else [])
        for path in paths:
            out = pk.paged_decode_attention(w.q.to(DEV), kc, vc, tables, ctx, lay.max_context_len, w.scale,
                                            err=err, path=path, window=window)
            torch.cuda.synchronize()
            assert err.item() == 0, (cfg, window, path)
            check_attention(out.double().cpu().numpy(), ref, w.q.dtype)
            checked += 1
    assert checked >= 8


@pytest.mark.parametrize("seed", [0, 1])
def test_random_shared_prefix_batches_match_oracle(seed):
    pk = require_gpu()
    rng = np.random.default_rng(6000 + seed)
    checked = 0
    for i in range(10):
        bs = int(rng.choice([16, 32, 64]))
        prefix = int(rng.integers(1, 60)) * bs
        G = int(rng.choice([1, 2, 3, 4, 6, 8]))
        cfg = configs.NANOCHAT.scaled(index=400 + seed * 100 + i, num_seqs=int(rng.integers(2, 40)),
                                      num_q_heads=8 * G, num_kv_heads=8, head_dim=int(rng.choice([64, 128])),
                                      block_size=bs, dtype=str(rng.choice(["bf16", "f16"])),
                                      ctx_args=(prefix, int(rng.choice([1, 5, 40, 300]))), vocab=1024)
        w = workloads.make_workload(cfg)
        lay = w.layout
        shared = pk.shared_prefix_len(lay.block_tables, lay.context_lens, bs)
        assert shared >= prefix
        kf, vf, _ = oracle_store_f64(w)
        ref = oracle.attention.decode_attention(w.q.double().numpy(), kf, vf, lay.block_tables, lay.context_lens,
                                                w.scale)
        cache = w.cache.to(DEV)
        kc, vc = cache[0, lay.layer], cache[1, lay.layer]
        tables = torch.from_numpy(lay.block_tables).to(DEV)
        ctx = torch.from_numpy(lay.context_lens).to(DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        slots = pk.slot_mapping(tables, ctx, bs, lay.num_blocks, err=err)
        pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, kc, vc, err=err)
        out = pk.paged_decode_attention_prefix(w.q.to(DEV), kc, vc, tables, ctx, lay.max_context_len, w.scale,
                                               prefix, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_attention(out.double().cpu().numpy(), ref, w.q.dtype)
        checked += 1
    assert checked == 10


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_sampler_rows_match_oracle(seed):
    pk = require_gpu()
    rng = np.random.default_rng(7000 + seed)
    exempt = rows = 0
    for _ in range(14):
        V = int(rng.choice([7, 100, 1000, 5000, 32000, 65536, 151936]))
        R = int(rng.integers(1, 64 if V <= 5000 else 12))
        dt = [torch.float32, torch.float16, torch.bfloat16][int(rng.integers(3))]
        x = torch.from_numpy((rng.standard_normal((R, V)) * float(rng.choice([0.5, 2.0, 3.0, 8.0]))).astype(np.float32))
        if rng.random() < 0.3:
            x = torch.round(x * 4) / 4                  # many ties
        x = x.to(dt)
        T = torch.from_numpy(rng.choice([0.0, 0.5, 1.0, 1.7], R).astype(np.float32))
        K = torch.from_numpy(rng.choice([0, 0, 1, 5, 50, 1000], R).astype(np.int32))
        P = torch.from_numpy(rng.choice([1.0, 1.0, 0.95, 0.9, 0.5, 0.1], R).astype(np.float32))
        S = torch.from_numpy(rng.integers(0, 2**62, R, dtype=np.int64))
        O = torch.from_numpy(rng.integers(0, 2**30, R, dtype=np.int64))
        tok = pk.sample(x.to(DEV), T.to(DEV), K.to(DEV), P.to(DEV), S.to(DEV), O.to(DEV)).cpu().numpy()
        for r in range(R):
            xr = x[r].double().numpy()
            rows += 1
            if float(T[r]) <= 0:
                assert int(tok[r]) == oracle.sampler.greedy(xr)
                continue
            ref, info = oracle.sampler.sample_row(xr, float(T[r]), int(K[r]), float(P[r]), int(S[r]), int(O[r]),
                                                  return_info=True)
            if int(tok[r]) != ref:
                assert sampling_exempt(info, float(P[r])), (V, str(dt), float(T[r]), int(K[r]), float(P[r]))
                exempt += 1
    assert exempt <= max(2, rows // 100)


@pytest.mark.parametrize("seed", [0, 1])
def test_random_prefill_batches_match_oracle(seed):
    """Varlen prefill (store bit-exact, attention on every (token, head)) over
    random head counts, groups up to 16, head_dim, block sizes 8-256, query
    lengths, cached prefixes (private or shared) and windows, on the
    tensor-core paths for 16-bit caches and the CUDA-core path for fp32."""
    from workloads import prefill as wp
    from test_gpu_prefill import oracle_cache, to_f64, run_prefill, check_rows
    from gpu_helpers import raw_numpy
    pk = require_gpu()
    rng = np.random.default_rng(8000 + seed)
    for i in range(8):
        dtype = str(rng.choice(["bf16", "f16", "f32"], p=[0.45, 0.45, 0.1]))
        hkv = int(rng.choice([1, 2, 4, 8]))
        B = int(rng.integers(1, 5))
        cfg = wp.PrefillConfig(name="random", index=600 + seed * 100 + i, num_seqs=B,
                               num_q_heads=hkv * int(rng.choice([1, 2, 3, 4, 6, 8, 16])), num_kv_heads=hkv,
                               head_dim=int(rng.choice([64, 128])), block_size=int(rng.choice([8, 16, 32, 64, 128, 256])),
                               dtype=dtype, q_kind="fixed",
                               q_args=tuple(int(x) for x in rng.integers(1, int(rng.choice([2, 40, 300])), B)),
                               hit_kind="fixed", hit_args=tuple(int(x) for x in rng.integers(0, 4, B)),
                               prefix_kind=str(rng.choice(["private", "shared"])))
        b = wp.make_prefill_batch(cfg)
        window = int(rng.choice([0, 0, 1, 33, 200]))
        k_ref, v_ref, slots_ref = oracle_cache(b)
        dt = b.cache.dtype
        ref = oracle.prefill.prefill_attention(b.q.double().numpy(), to_f64(k_ref, dt), to_f64(v_ref, dt),
                                               b.block_tables, b.cu_seqlens_q, b.cu_seqlens_k, b.scale, window=window)
        T, Hq, _ = ref.shape
        for path in (["fma"] if dtype == "f32" else ["tc", "mma"]):
            cache, slots, out, err = run_prefill(pk, b, window=window,
                                                 path={"tc": pk.PATH_TC, "mma": pk.PATH_MMA, "fma": pk.PATH_FMA}[path])
            assert err == 0, (cfg, window, path)
            np.testing.assert_array_equal(slots, slots_ref)
            np.testing.assert_array_equal(raw_numpy(cache[0]), k_ref)
            np.testing.assert_array_equal(raw_numpy(cache[1]), v_ref)
            check_rows(out.double().numpy(), ref, [(t, h) for t in range(T) for h in range(Hq)], f32=dtype == "f32")


@pytest.mark.parametrize("seed", [0, 1])
def test_random_sample_ex_rows_match_oracle(seed):
    """The sampler extras over random vocabularies (16-byte rows, which a
    mask needs), dtypes, masks from all-allowed to nearly-all-masked, and cut
    parameters: ids, token_prob and the top-8 against the oracle."""
    pk = require_gpu()
    rng = np.random.default_rng(9000 + seed)
    for _ in range(10):
        V = int(rng.choice([8, 96, 1000, 5000, 32000, 65536, 151936]))
        R = int(rng.integers(1, 32 if V <= 5000 else 8))
        dt = [torch.float32, torch.float16, torch.bfloat16][int(rng.integers(3))]
        x = (rng.standard_normal((R, V)) * float(rng.choice([0.5, 2.0, 3.0, 8.0]))).astype(np.float32)
        if rng.random() < 0.3:
            x = np.round(x * 4) / 4
        logits = torch.from_numpy(x).to(dt)
        T = rng.choice([0.0, 0.6, 1.0, 1.4], R).astype(np.float32)
        K = rng.choice([0, 1, 5, 50, 300], R).astype(np.int32)
        P = rng.choice([1.0, 0.95, 0.9, 0.5], R).astype(np.float32)
        allowed = rng.random((R, V)) > rng.choice([0.0, 0.0, 0.3, 0.9, 0.999], R)[:, None]
        S = rng.integers(0, 2**62, R, dtype=np.int64)
        O = rng.integers(0, 2**30, R, dtype=np.int64)
        tok, tp, p8, i8 = pk.sample_ex(logits.to(DEV), torch.from_numpy(T).to(DEV), torch.from_numpy(K).to(DEV),
                                       torch.from_numpy(P).to(DEV), torch.from_numpy(S).to(DEV),
                                       torch.from_numpy(O).to(DEV), mask_words=pk.pack_mask(torch.from_numpy(allowed)).to(DEV))
        tok, tp, p8, i8 = tok.cpu().numpy(), tp.cpu().numpy(), p8.cpu().numpy(), i8.cpu().numpy()
        xd = logits.double().numpy()
        for r in range(R):
            if not allowed[r].any():
                assert 0 <= tok[r] < V
                continue
            (rt, rp, r8p, r8i), info = oracle.sampler.sample_outputs(xd[r], float(T[r]), int(K[r]), float(P[r]),
                                                                      int(S[r]), int(O[r]), mask=allowed[r],
                                                                      return_info=True)
            if int(tok[r]) != rt:
                assert sampling_exempt(info, float(P[r]))
                continue
            assert allowed[r, tok[r]]
            np.testing.assert_allclose(tp[r], rp, rtol=1e-5, atol=1e-30)
            nv = min(8, V)
            assert i8[r][:nv].tolist() == r8i[:nv].tolist()
            np.testing.assert_allclose(p8[r][:nv], r8p[:nv], rtol=1e-5, atol=1e-30)
