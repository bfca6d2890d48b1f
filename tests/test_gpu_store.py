"""Slot mapping and KV store on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import configs
from gpu_helpers import require_gpu, raw_numpy, oracle_store_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", list(configs.CONFIGS))
def test_slot_mapping_all_configs(name):
    pk = require_gpu()
    cfg = configs.CONFIGS[name]
    lay = workloads.make_layout(cfg)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = pk.slot_mapping(torch.from_numpy(lay.block_tables).to(DEV),
                          torch.from_numpy(lay.context_lens).to(DEV), cfg.block_size,
                          lay.num_blocks, err=err)
    ref = oracle.paging.decode_slot_mapping(lay.block_tables, lay.context_lens, cfg.block_size)
    assert np.array_equal(got.cpu().numpy(), ref)
    assert err.item() == 0


def test_slot_mapping_edge_cases_and_flags():
    pk = require_gpu()
    tables = torch.tensor([[5, 10, -1], [7, -1, -1], [3, 99, 2], [2, 0, 1], [4, 6, 8]],
                          dtype=torch.int32, device=DEV)
    ctx = torch.tensor([300, 0, 400, 769, 1], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = pk.slot_mapping(tables, ctx, 256, 64, err=err).cpu().tolist()
    # row 2: block id 99 >= 64 -> flagged, -1 ; row 3: position 768 needs a 4th block -> flagged
    assert got == [10 * 256 + 43, -1, -1, -1, 4 * 256]
    assert err.item() == (pk.ERR_BLOCK_ID | pk.ERR_CONTEXT)


def _small_variants():
    return {
        "tiny": configs.TINY,
        "nanochat": configs.NANOCHAT,
        "qwen3_small": configs.QWEN3.scaled(num_seqs=5, ctx_args=(1, 600), pool_blocks=40, num_layers=3,
                                            vocab=2048),
        "grok1_small": configs.GROK1.scaled(num_seqs=3, ctx_args=(77,), vocab=2048),
        "longctx_small": configs.LONGCTX.scaled(num_seqs=5, ctx_args=(1, 700), vocab=2048),
    }


@pytest.mark.parametrize("name", list(_small_variants()))
def test_kv_store_bit_exact(name):
    pk = require_gpu()
    cfg = _small_variants()[name]
    w = workloads.make_workload(cfg)
    lay = w.layout
    cache = w.cache.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = pk.slot_mapping(torch.from_numpy(lay.block_tables).to(DEV),
                            torch.from_numpy(lay.context_lens).to(DEV), cfg.block_size, lay.num_blocks)
    pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, cache[0, lay.layer], cache[1, lay.layer], err=err)
    _, _, ref_slots = oracle_store_f64(w)
    k = raw_numpy(w.k_cache())
    v = raw_numpy(w.v_cache())
    oracle.store.kv_store(raw_numpy(w.k_new), raw_numpy(w.v_new), ref_slots, k, v)
    got = cache.cpu()
    assert np.array_equal(raw_numpy(got[0, lay.layer]), k)
    assert np.array_equal(raw_numpy(got[1, lay.layer]), v)
    # other layers of a multi-layer cache are untouched
    for l in range(cfg.num_layers):
        if l != lay.layer:
            assert np.array_equal(raw_numpy(got[:, l]), raw_numpy(w.cache[:, l]))
    assert err.item() == 0


def test_kv_store_skips_negative_and_flags_out_of_range():
    pk = require_gpu()
    nb, bs, H, D = 8, 16, 2, 64
    kc = torch.zeros(nb, bs, H, D, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.randn(3, H, D, device=DEV).to(torch.bfloat16)
    k.view(torch.int16)[0, 0, 0] = 0x7FC1            # NaN payload survives a bit copy
    v = torch.randn(3, H, D, device=DEV).to(torch.bfloat16)
    slots = torch.tensor([17, -1, nb * bs], dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk.kv_store(k, v, slots, kc, vc, err=err)
    assert torch.equal(kc[1, 1].view(torch.int16), k[0].view(torch.int16))
    assert torch.equal(vc[1, 1].view(torch.int16), v[0].view(torch.int16))
    mask = torch.ones(nb, bs, dtype=torch.bool, device=DEV)
    mask[1, 1] = False
    assert torch.all(kc[mask].view(torch.int16) == 0)
    assert err.item() == pk.ERR_SLOT


FULL = {"qwen3_full": configs.QWEN3, "grok1_full": configs.GROK1, "longctx_full": configs.LONGCTX}


def _touched_blocks(lay, bs):
    """Rows with a token to store, the block each one's slot falls in, and the
    row offset inside that block."""
    ctx = lay.context_lens.astype(np.int64)
    rows = np.nonzero(ctx > 0)[0]
    blocks = np.array([lay.block_tables[i, (ctx[i] - 1) // bs] for i in rows], dtype=np.int64)
    return rows, blocks, (ctx[rows] - 1) % bs


@pytest.mark.parametrize("name", list(_small_variants()) + list(FULL))
def test_kv_store_paged_matches_the_two_step_store(name):
    """The fused slot-mapping + store kernel writes the same cache bits and
    slots as pkvd_slot_mapping followed by pkvd_kv_store, and the blocks it
    touches hold what the oracle's store writes into a copy of them."""
    pk = require_gpu()
    cfg = FULL[name] if name in FULL else _small_variants()[name]
    w = workloads.make_workload(cfg, device=DEV if name in FULL else "cpu")
    lay = w.layout
    base = w.cache.to(DEV)
    # the oracle's store on a host copy of every block the step writes into
    rows, blocks, offs = _touched_blocks(lay, cfg.block_size)
    bidx = torch.from_numpy(blocks).to(DEV)
    k_ref = raw_numpy(base[0, lay.layer].index_select(0, bidx).cpu())
    v_ref = raw_numpy(base[1, lay.layer].index_select(0, bidx).cpu())
    sub_slots = np.arange(len(rows), dtype=np.int64) * cfg.block_size + offs
    ridx = torch.from_numpy(rows)
    oracle.store.kv_store(raw_numpy(w.k_new.cpu()[ridx]), raw_numpy(w.v_new.cpu()[ridx]), sub_slots, k_ref, v_ref)
    tables = torch.from_numpy(lay.block_tables).to(DEV)
    ctx = torch.from_numpy(lay.context_lens).to(DEV)
    k_new, v_new = w.k_new.to(DEV), w.v_new.to(DEV)
    two = base.clone()
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots2 = pk.slot_mapping(tables, ctx, cfg.block_size, lay.num_blocks, err=err2)
    pk.kv_store(k_new, v_new, slots2, two[0, lay.layer], two[1, lay.layer], err=err2)
    one = base
    err1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots1 = torch.full_like(slots2, 12345)
    pk.kv_store_paged(k_new, v_new, tables, ctx, one[0, lay.layer], one[1, lay.layer], slot_mapping=slots1, err=err1)
    torch.cuda.synchronize()
    assert torch.equal(slots1, slots2)
    assert torch.equal(one.view(torch.int16) if one.dtype != torch.float32 else one.view(torch.int32),
                       two.view(torch.int16) if two.dtype != torch.float32 else two.view(torch.int32))
    assert err1.item() == 0 and err2.item() == 0
    ref = oracle.paging.decode_slot_mapping(lay.block_tables, lay.context_lens, cfg.block_size)
    assert np.array_equal(slots1.cpu().numpy(), ref)
    assert np.array_equal(raw_numpy(one[0, lay.layer].index_select(0, bidx).cpu()), k_ref)
    assert np.array_equal(raw_numpy(one[1, lay.layer].index_select(0, bidx).cpu()), v_ref)


def test_kv_store_paged_flags_and_skips_like_slot_mapping():
    pk = require_gpu()
    tables = torch.tensor([[5, 10, -1], [7, -1, -1], [3, 99, 2], [2, 0, 1], [4, 6, 8]],
                          dtype=torch.int32, device=DEV)
    ctx = torch.tensor([300, 0, 400, 769, 1], dtype=torch.int32, device=DEV)
    nb, bs, H, D = 64, 256, 1, 64
    kc = torch.zeros(nb, bs, H, D, dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.randn(5, H, D, device=DEV).to(torch.float16)
    v = torch.randn(5, H, D, device=DEV).to(torch.float16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = torch.empty(5, dtype=torch.int64, device=DEV)
    pk.kv_store_paged(k, v, tables, ctx, kc, vc, slot_mapping=slots, err=err)
    assert slots.cpu().tolist() == [10 * 256 + 43, -1, -1, -1, 4 * 256]
    assert err.item() == (pk.ERR_BLOCK_ID | pk.ERR_CONTEXT)
    assert torch.equal(kc[10, 43, 0], k[0, 0]) and torch.equal(vc[4, 0, 0], v[4, 0])
    written = torch.zeros(nb, bs, dtype=torch.bool, device=DEV)
    written[10, 43] = True
    written[4, 0] = True
    assert torch.all(kc[~written] == 0) and torch.all(vc[~written] == 0)
    # no slot output requested: same cache writes
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    pk.kv_store_paged(k, v, tables, ctx, kc2, vc2)
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)


@pytest.mark.parametrize("dtype,H,D,bs", [(torch.float16, 16, 64, 256), (torch.bfloat16, 8, 128, 16),
                                          (torch.float32, 2, 64, 16)])
def test_copy_blocks_copies_the_leading_rows_bit_exactly(dtype, H, D, bs):
    pk = require_gpu()
    nb = 40
    g = torch.Generator(device="cpu").manual_seed(8)
    kc = torch.randn(nb, bs, H, D, generator=g).to(dtype).to(DEV)
    vc = torch.randn(nb, bs, H, D, generator=g).to(dtype).to(DEV)
    src = torch.tensor([3, 7, 11, 0], dtype=torch.int32)
    dst = torch.tensor([20, 21, 22, 23], dtype=torch.int32)
    rows = torch.tensor([bs - 1, 1, 0, bs], dtype=torch.int32)
    k0, v0 = kc.clone(), vc.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pk.copy_blocks(kc, vc, src.to(DEV), dst.to(DEV), rows.to(DEV), err=err)
    torch.cuda.synchronize()
    ek, ev = k0.clone(), v0.clone()
    for s_, d_, r_ in zip(src.tolist(), dst.tolist(), rows.tolist()):
        ek[d_, :r_] = k0[s_, :r_]
        ev[d_, :r_] = v0[s_, :r_]
    assert torch.equal(kc, ek) and torch.equal(vc, ev) and err.item() == 0
    bad = torch.tensor([nb], dtype=torch.int32, device=DEV)
    pk.copy_blocks(kc, vc, bad, dst[:1].to(DEV), rows[:1].to(DEV), err=err)
    torch.cuda.synchronize()
    assert err.item() == pk.ERR_BLOCK_ID and torch.equal(kc, ek)


def test_block_manager_fork_and_copy_on_write_on_the_device():
    """Two clones of a prompt share its blocks; each decodes its own token into
    the shared partial block after the copy-on-write copy, and attention over
    either sequence equals the oracle over that sequence's own K/V."""
    pk = require_gpu()
    import oracle as orc
    nb, bs, H, D, G = 16, 16, 2, 64, 2
    g = torch.Generator(device="cpu").manual_seed(9)
    kc = torch.full((nb, bs, H, D), float("nan"), dtype=torch.float16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    bm = pk.BlockManager(nb, bs)
    prompt = list(range(100, 137))                            # 37 tokens: blocks 0, 1 full, 2 partial
    table, cached = bm.allocate(prompt)
    assert cached == 0
    kv = {p: (torch.randn(H, D, generator=g).half(), torch.randn(H, D, generator=g).half()) for p in range(40)}
    for p in range(len(prompt)):                              # the prompt's K/V rows, through the store kernel
        t_ = torch.tensor([table + [-1] * 2], dtype=torch.int32, device=DEV)
        pk.kv_store_paged(kv[p][0].unsqueeze(0).to(DEV), kv[p][1].unsqueeze(0).to(DEV), t_,
                          torch.tensor([p + 1], dtype=torch.int32, device=DEV), kc, vc)
    clone = bm.fork(table)
    seqs = {"a": (prompt + [1], table), "b": (prompt + [2], clone)}
    own = {"a": torch.randn(H, D, generator=g).half(), "b": torch.randn(H, D, generator=g).half()}
    q = torch.randn(2, H * G, D, generator=g).half()
    outs, tabs = {}, {}
    for name, (toks, tab) in seqs.items():
        t2, cp = bm.append(toks, tab)
        if cp is not None:
            pk.copy_blocks(kc, vc, *(torch.tensor([x], dtype=torch.int32, device=DEV) for x in cp))
        tabs[name] = t2
        tt = torch.tensor([t2 + [-1] * 2], dtype=torch.int32, device=DEV)
        ctx = torch.tensor([len(toks)], dtype=torch.int32, device=DEV)
        pk.kv_store_paged(own[name].unsqueeze(0).to(DEV), own[name].unsqueeze(0).to(DEV), tt, ctx, kc, vc)
    # the first clone copied the shared partial block; the second then owned the original alone
    assert tabs["a"][:2] == table[:2] and tabs["a"][2] != table[2] and tabs["b"] == table
    for i, name in enumerate(["a", "b"]):
        toks, _ = seqs[name]
        tt = torch.tensor([tabs[name] + [-1] * 2], dtype=torch.int32, device=DEV)
        ctx = torch.tensor([len(toks)], dtype=torch.int32, device=DEV)
        out = pk.paged_decode_attention(q[i:i + 1].to(DEV), kc, vc, tt, ctx, len(toks), 0.125)
        K = torch.stack([kv[p][0] for p in range(len(prompt))] + [own[name]]).double().numpy()
        V = torch.stack([kv[p][1] for p in range(len(prompt))] + [own[name]]).double().numpy()
        kc_ref = K[:, None]                                   # [ctx, 1(row), H, D] as one-row blocks
        ref = orc.attention.decode_attention(q[i:i + 1].double().numpy(), kc_ref, V[:, None],
                                             np.arange(len(toks))[None, :], np.array([len(toks)]), 0.125)
        rel = (out.double().cpu().numpy() - ref).__abs__().max() / np.abs(ref).max()
        assert rel < 2e-2 and torch.isfinite(out).all()
