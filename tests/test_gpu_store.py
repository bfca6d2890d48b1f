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
