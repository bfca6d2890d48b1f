"""The graph-captured decode step gives the same results as the eager calls."""
import numpy as np
import pytest
import torch

import workloads
from workloads import configs
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", ["tiny", "nanochat", "grok1"])
def test_graph_replay_matches_eager(name):
    pk = require_gpu()
    cfg = configs.CONFIGS[name]
    w = workloads.make_workload(cfg, device=DEV if name == "grok1" else "cpu")
    lay = w.layout
    cache = w.cache.to(DEV)
    kc, vc = cache[0, lay.layer], cache[1, lay.layer]
    step = pk.DecodeStep(kc, vc, lay.num_seqs, cfg.num_q_heads, lay.max_blocks_per_seq,
                         lay.max_context_len, cfg.vocab, w.logits.dtype, w.scale)
    step.q.copy_(w.q)
    step.k_new.copy_(w.k_new)
    step.v_new.copy_(w.v_new)
    step.block_tables.copy_(torch.from_numpy(lay.block_tables))
    step.context_lens.copy_(torch.from_numpy(lay.context_lens))
    step.logits.copy_(w.logits)
    step.temperature.copy_(torch.from_numpy(w.temperature))
    step.top_k.copy_(torch.from_numpy(w.top_k))
    step.top_p.copy_(torch.from_numpy(w.top_p))
    step.seeds.copy_(torch.from_numpy(w.seeds.view(np.int64)))
    step.enqueue()
    torch.cuda.synchronize()
    out_eager, tok_eager = step.out.clone(), step.token_ids.clone()
    # eager equals the individual binding calls
    tables = step.block_tables
    ctx = step.context_lens
    out2 = pk.paged_decode_attention(step.q, kc, vc, tables, ctx, lay.max_context_len, w.scale)
    tok2 = pk.sample(step.logits, step.temperature, step.top_k, step.top_p, step.seeds, step.offsets)
    assert torch.equal(out2, out_eager) and torch.equal(tok2, tok_eager)
    step.capture()
    step.out.zero_()
    step.token_ids.fill_(-1)
    for _ in range(3):
        step.replay()
    torch.cuda.synchronize()
    assert torch.equal(step.out, out_eager)
    assert torch.equal(step.token_ids, tok_eager)
    # a new step's inputs flow through the same graph
    step.offsets.add_(1)
    step.replay()
    tok3 = pk.sample(step.logits, step.temperature, step.top_k, step.top_p, step.seeds, step.offsets)
    torch.cuda.synchronize()
    assert torch.equal(step.token_ids, tok3)
    assert step.err.item() == 0
