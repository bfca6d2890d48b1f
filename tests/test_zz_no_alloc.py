"""The allocation-free attention entry point.

pkvd_paged_decode_attention_noalloc serves callers that cannot allocate
device memory where they call (engines whose paged KV cache took all free
memory at start-up, plugins in a runtime that owns every allocation, loops
that must not synchronise on cudaMalloc, plain C hosts): it runs the same
attention on a scratch array built into the library.  Here it is called through the C ABI and compared,
on two calls in a row, with the regular entry point that takes a workspace.
This file is collected last so that a failure here leaves every other test
already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from workloads import configs
from gpu_helpers import require_gpu, check_attention

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(cfg):
    pk = require_gpu()
    w = workloads.make_workload(cfg)
    lay = w.layout
    cache = w.cache.to(DEV)
    kc, vc = cache[0, lay.layer], cache[1, lay.layer]
    tables = torch.from_numpy(lay.block_tables).to(DEV)
    ctx = torch.from_numpy(lay.context_lens).to(DEV)
    slots = pk.slot_mapping(tables, ctx, cfg.block_size, lay.num_blocks)
    pk.kv_store(w.k_new.to(DEV), w.v_new.to(DEV), slots, kc, vc)
    return pk, w, lay, kc, vc, tables, ctx


def _call_noalloc(pk, q, kc, vc, tables, ctx, lay, scale, out, err):
    from paged_kv_decode_store_gb300 import _capi
    c = _capi.cache_desc(kc, vc)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return pk.lib().pkvd_paged_decode_attention_noalloc(
        out.data_ptr(), q.data_ptr(), ctypes.byref(c), tables.data_ptr(), tables.shape[1], ctx.data_ptr(),
        lay.max_context_len, lay.num_seqs, q.shape[1], ctypes.c_float(scale), stream, err.data_ptr())


@pytest.mark.parametrize("cfg", [configs.GROK1.scaled(num_seqs=9, ctx_kind="explicit",
                                                      ctx_args=(700, 1, 0, 333, 2048, 17, 1500, 64, 999),
                                                      table_kind="perm", vocab=2048),
                                 configs.NANOCHAT],
                         ids=["grok1_ragged", "nanochat"])
def test_noalloc_matches_workspace_entry_point_twice(cfg):
    pk, w, lay, kc, vc, tables, ctx = _inputs(cfg)
    q = w.q.to(DEV)
    for _ in range(2):                             # the scratch keeps the last call's contents
        ref = pk.paged_decode_attention(q, kc, vc, tables, ctx, lay.max_context_len, w.scale)
        out = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _call_noalloc(pk, q, kc, vc, tables, ctx, lay, w.scale, out, err) == 0
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.isfinite(out).all()
        check_attention(out.double().cpu().numpy(), ref.double().cpu().numpy(), q.dtype)


def _big_call(pk, entry, kc, vc, num_heads, scale, ws=None):
    """A call with 4096 rows of `num_heads` query heads on buffers sized for it
    (so even a call that went through would stay in bounds)."""
    from paged_kv_decode_store_gb300 import _capi
    B, D = 4096, kc.shape[-1]
    q = torch.zeros(B, num_heads, D, dtype=kc.dtype, device=DEV)
    out = torch.empty_like(q)
    tables = torch.zeros(B, 4, dtype=torch.int32, device=DEV)
    ctx = torch.full((B,), 64, dtype=torch.int32, device=DEV)
    c = _capi.cache_desc(kc, vc)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [out.data_ptr(), q.data_ptr(), ctypes.byref(c), tables.data_ptr(), 4, ctx.data_ptr(), 64, B,
            num_heads, ctypes.c_float(scale)]
    if entry == "noalloc":
        st = pk.lib().pkvd_paged_decode_attention_noalloc(*args, stream, err.data_ptr())
    else:
        st = pk.lib().pkvd_paged_decode_attention(*args, ws.data_ptr(), ws.numel(), stream, err.data_ptr())
    torch.cuda.synchronize()
    return st, err.item()


def test_every_supported_shape_fits_the_scratch_on_this_gpu():
    """The scratch limit (16 MiB) is checked after the argument checks, so only
    a supported shape can reach it.  On this GPU none does: the largest
    workspace of any supported head layout is below the limit (the check can
    only trigger on GPUs with many more SMs), so every supported call runs."""
    pk = require_gpu()
    # the supported layouts with the most query heads x (head_dim + 4): 8 KV
    # heads of 128 and 16 KV heads of 64, each with groups of 8
    largest = max(pk.decode_workspace_bytes(4096, 64, 128, 32768), pk.decode_workspace_bytes(4096, 128, 64, 32768))
    assert 0 < largest <= 16 << 20
    # the limit does bind for a GPU four times this size (same shapes, more SMs)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = ctypes.c_size_t(0)
    assert pk.lib().pkvd_decode_workspace_bytes(4096, 64, 128, 32768, 4 * sms, ctypes.byref(n)) == 0
    assert n.value > 16 << 20


@pytest.mark.parametrize("heads,scale,status", [(132, 0.1, 3), (128, float("inf"), 1)],
                         ids=["group_not_dividing", "scale_not_finite"])
def test_noalloc_reports_invalid_calls_like_the_workspace_entry_point(heads, scale, status):
    """An invalid call that is also too big for the scratch gets the workspace
    entry point's status (the shape or argument error), not the size error."""
    pk, w, lay, kc, vc, tables, ctx = _inputs(configs.GROK1.scaled(num_seqs=2, ctx_args=(64,), vocab=2048))
    ws = torch.zeros(32 << 20, dtype=torch.uint8, device=DEV)
    st_ws, _ = _big_call(pk, "workspace", kc, vc, heads, scale, ws)
    st_na, err = _big_call(pk, "noalloc", kc, vc, heads, scale)
    assert st_ws == status and st_na == status and err == 0
