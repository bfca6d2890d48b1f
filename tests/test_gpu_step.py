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


def test_host_staged_step_matches_device_step():
    """replay_host(): inputs from pinned host arenas, logits copied beside the
    store and attention kernels, outputs copied back -- same results."""
    pk = require_gpu()
    cfg = configs.NANOCHAT
    w = workloads.make_workload(cfg)
    lay = w.layout
    cache = w.cache.to(DEV)
    kc, vc = cache[0, lay.layer], cache[1, lay.layer]
    step = pk.DecodeStep(kc, vc, lay.num_seqs, cfg.num_q_heads, lay.max_blocks_per_seq,
                         lay.max_context_len, cfg.vocab, w.logits.dtype, w.scale)
    host = {"q": w.q, "k_new": w.k_new, "v_new": w.v_new, "block_tables": torch.from_numpy(lay.block_tables),
            "context_lens": torch.from_numpy(lay.context_lens), "logits": w.logits,
            "temperature": torch.from_numpy(w.temperature), "top_k": torch.from_numpy(w.top_k),
            "top_p": torch.from_numpy(w.top_p), "seeds": torch.from_numpy(w.seeds.view(np.int64)),
            "offsets": torch.from_numpy(w.offsets.view(np.int64))}
    h = step.host_buffers()
    for k, t in host.items():
        h[k].copy_(t)
    step.replay_host()
    torch.cuda.synchronize()
    out_h, tok_h = h["out"].clone(), h["token_ids"].clone()
    # the same inputs through the device buffers (cache rows are rewritten
    # with the same values, so a second pass sees the same cache)
    for k, t in host.items():
        getattr(step, k).copy_(t)
    step.enqueue()
    torch.cuda.synchronize()
    assert torch.equal(out_h, step.out.cpu())
    assert torch.equal(tok_h, step.token_ids.cpu())
    # a changed host input reaches the device through the graph
    h["offsets"].add_(7)
    step.replay_host()
    torch.cuda.synchronize()
    assert torch.equal(step.offsets.cpu(), h["offsets"])       # copied in by the step
    tok_ref = pk.sample(step.logits, step.temperature, step.top_k, step.top_p, step.seeds, step.offsets)
    torch.cuda.synchronize()
    assert torch.equal(h["token_ids"], tok_ref.cpu())
    assert step.err.item() == 0


def test_step_with_sampler_extras_matches_the_eager_calls():
    pk = require_gpu()
    cfg = configs.NANOCHAT
    w = workloads.make_workload(cfg, device=DEV)
    lay = w.layout
    kc, vc = w.cache[0, lay.layer], w.cache[1, lay.layer]
    step = pk.DecodeStep(kc, vc, lay.num_seqs, cfg.num_q_heads, lay.max_blocks_per_seq,
                         lay.max_context_len, cfg.vocab, w.logits.dtype, w.scale, extras=True)
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
    g = torch.Generator().manual_seed(3)
    step.mask_words.copy_(pk.pack_mask(torch.rand(lay.num_seqs, cfg.vocab, generator=g) > 0.2))
    step.capture()
    step.replay()
    torch.cuda.synchronize()
    tok, tp, p8, i8 = pk.sample_ex(step.logits, step.temperature, step.top_k, step.top_p, step.seeds,
                                   step.offsets, mask_words=step.mask_words)
    torch.cuda.synchronize()
    assert torch.equal(step.token_ids, tok) and torch.equal(step.token_prob, tp)
    assert torch.equal(step.top_probs, p8) and torch.equal(step.top_ids, i8)
    assert step.kernels_per_step == 5 and step.err.item() == 0
