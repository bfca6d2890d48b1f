"""One decode step for one layer, as a fixed-shape CUDA graph.

nano-vllm "Model Runner" notes, section "run model": the decode shape is
fixed (one token per sequence), so the step is captured once and replayed,
saving the per-kernel launch cost that Grok-1 "第 8 章 runners.py 推理引擎"
section 8.7 lists among its decode slowdowns.  Every per-step value (block
tables, context lengths, sampling parameters, Philox offsets) lives in a
device buffer owned by this object; a step is: write the inputs into those
buffers, replay.

Step order (all library kernels):
    slot_mapping -> kv_store -> paged_decode_attention (partition + merge) -> sample
"""
from __future__ import annotations

import ctypes

import torch

from . import _capi


class DecodeStep:
    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, num_seqs: int,
                 num_q_heads: int, max_blocks_per_seq: int, max_context_len: int,
                 vocab: int, logits_dtype: torch.dtype, scale: float,
                 path: int = _capi.PATH_AUTO):
        dev = k_cache.device
        nb, bs, Hkv, D = k_cache.shape
        B, Hq = num_seqs, num_q_heads
        self.k_cache, self.v_cache = k_cache, v_cache
        self.B, self.Hq, self.Hkv, self.D, self.bs, self.nb = B, Hq, Hkv, D, bs, nb
        self.max_context_len = max_context_len
        self.scale = float(scale)
        self.path = path
        dt = k_cache.dtype
        self.q = torch.zeros(B, Hq, D, dtype=dt, device=dev)
        self.k_new = torch.zeros(B, Hkv, D, dtype=dt, device=dev)
        self.v_new = torch.zeros(B, Hkv, D, dtype=dt, device=dev)
        self.block_tables = torch.full((B, max_blocks_per_seq), -1, dtype=torch.int32, device=dev)
        self.context_lens = torch.zeros(B, dtype=torch.int32, device=dev)
        self.slots = torch.empty(B, dtype=torch.int64, device=dev)
        self.out = torch.empty(B, Hq, D, dtype=dt, device=dev)
        self.logits = torch.zeros(B, vocab, dtype=logits_dtype, device=dev)
        self.temperature = torch.ones(B, dtype=torch.float32, device=dev)
        self.top_k = torch.zeros(B, dtype=torch.int32, device=dev)
        self.top_p = torch.ones(B, dtype=torch.float32, device=dev)
        self.seeds = torch.zeros(B, dtype=torch.int64, device=dev)
        self.offsets = torch.zeros(B, dtype=torch.int64, device=dev)
        self.token_ids = torch.empty(B, dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        nbytes = ctypes.c_size_t(0)
        _capi.check(_capi.lib().pkvd_decode_workspace_bytes(B, Hq, D, max_context_len, 0,
                                                            ctypes.byref(nbytes)))
        self.workspace = torch.zeros(max(int(nbytes.value), 16), dtype=torch.uint8, device=dev)
        self.cache = _capi.cache_desc(k_cache, v_cache)
        self.graph = None
        self.kernels_per_step = 5     # slot, store, partition, merge, sample

    def enqueue(self, stream=None) -> None:
        L = _capi.lib()
        s = _capi.stream_handle(stream, self.q)
        p = _capi.ptr
        _capi.check(L.pkvd_slot_mapping(p(self.slots), p(self.block_tables), self.block_tables.shape[1],
                                        p(self.context_lens), self.B, self.bs, self.nb, s, p(self.err)))
        _capi.check(L.pkvd_kv_store(p(self.k_new), p(self.v_new), p(self.slots), self.B,
                                    ctypes.byref(self.cache), s, p(self.err)))
        _capi.check(L.pkvd_paged_decode_attention_ex(
            p(self.out), p(self.q), ctypes.byref(self.cache), p(self.block_tables),
            self.block_tables.shape[1], p(self.context_lens), self.max_context_len, self.B, self.Hq,
            ctypes.c_float(self.scale), p(self.workspace), self.workspace.numel(), s, p(self.err),
            self.path))
        V = self.logits.shape[1]
        _capi.check(L.pkvd_sample(p(self.token_ids), p(self.logits), _capi.dtype_code(self.logits.dtype),
                                  self.B, V, self.logits.stride(0), p(self.temperature), p(self.top_k),
                                  p(self.top_p), p(self.seeds), p(self.offsets), None, 0, s))

    def capture(self) -> None:
        """Record the step into a CUDA graph (after one eager warm-up run)."""
        side = torch.cuda.Stream(device=self.q.device)
        side.wait_stream(torch.cuda.current_stream(self.q.device))
        with torch.cuda.stream(side):
            self.enqueue()
        torch.cuda.current_stream(self.q.device).wait_stream(side)
        torch.cuda.synchronize(self.q.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.enqueue()
        self.graph = g

    def replay(self) -> None:
        if self.graph is None:
            self.enqueue()
        else:
            self.graph.replay()
