"""The seeded generator produces the structures the five workloads name."""
import numpy as np
import torch

import workloads
from workloads import configs


def test_layouts_have_named_structure():
    for cfg in configs.CONFIGS.values():
        lay = workloads.make_layout(cfg)
        ctx, tab = lay.context_lens, lay.block_tables
        assert ctx.shape == (cfg.num_seqs,)
        bs = cfg.block_size
        used = []
        for i, c in enumerate(ctx):
            n = -(-int(c) // bs)
            assert np.all(tab[i, :n] >= 0) and np.all(tab[i, n:] == -1)
            assert np.all(tab[i, :n] < lay.num_blocks)
            used.extend(tab[i, :n].tolist())
        if cfg.table_kind != "shared_prefix":
            assert len(used) == len(set(used))       # no block shared
        assert ctx.max() <= lay.max_context_len
    tiny = workloads.make_layout(configs.TINY)
    assert tiny.context_lens.tolist() == [1, 17, 33, 50] and tiny.num_blocks == 32
    g = workloads.make_layout(configs.GROK1)
    assert np.array_equal(g.block_tables[3], np.arange(3 * 128, 4 * 128))
    n = workloads.make_layout(configs.NANOCHAT)
    assert np.all(n.block_tables[:, :64] == n.block_tables[0, :64])   # shared prefix blocks
    assert np.all((n.context_lens >= 1025) & (n.context_lens <= 1280))
    q = workloads.make_layout(configs.QWEN3)
    assert q.num_blocks == 1024 and 0 <= q.layer < 28
    assert np.all((q.context_lens >= 128) & (q.context_lens <= 4096))
    l5 = workloads.make_layout(configs.LONGCTX)
    assert np.all((l5.context_lens >= 512) & (l5.context_lens <= 32768))


def test_seeded_and_poisoned():
    a = workloads.make_workload(configs.TINY)
    b = workloads.make_workload(configs.TINY)
    assert torch.equal(a.q, b.q) and torch.equal(a.logits, b.logits)
    kc = a.k_cache()
    lay = a.layout
    # rows at/after the new token in each last block are NaN; earlier rows are finite
    for i, c in enumerate(lay.context_lens):
        c = int(c)
        last = lay.block_tables[i, (c - 1) // 16]
        r = (c - 1) % 16
        assert torch.isnan(kc[last, r:]).all()
        assert torch.isfinite(kc[last, :r]).all()
    used = set(lay.block_tables[lay.block_tables >= 0].tolist())
    for blk in range(lay.num_blocks):
        if blk not in used:
            assert torch.isnan(kc[blk]).all()
