"""One decode step for one layer, as a fixed-shape CUDA graph.

nano-vllm "Model Runner" notes, section "run model": the decode shape is
fixed (one token per sequence), so the step is captured once and replayed,
saving the per-kernel launch cost that Grok-1 "第 8 章 runners.py 推理引擎"
section 8.7 lists among its decode slowdowns.  Every per-step value (block
tables, context lengths, sampling parameters, Philox offsets) lives in a
device buffer owned by this object; a step is: write the inputs into those
buffers, replay.

Step order (all library kernels):
    kv_store_paged (slot mapping + store) -> paged_decode_attention (partition + merge) -> sample
(paged_decode_attention_prefix instead when the rows share a cached prefix,
nanochat's one prefill cloned N ways).
"""
from __future__ import annotations

import ctypes

import torch

from . import _capi


class DecodeStep:
    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, num_seqs: int,
                 num_q_heads: int, max_blocks_per_seq: int, max_context_len: int,
                 vocab: int, logits_dtype: torch.dtype, scale: float,
                 path: int = _capi.PATH_AUTO, window: int = 0, extras: bool = False,
                 shared_prefix_len: int = 0):
        dev = k_cache.device
        nb, bs, Hkv, D = k_cache.shape
        B, Hq = num_seqs, num_q_heads
        self.k_cache, self.v_cache = k_cache, v_cache
        self.B, self.Hq, self.Hkv, self.D, self.bs, self.nb = B, Hq, Hkv, D, bs, nb
        self.max_context_len = max_context_len
        self.scale = float(scale)
        self.path = path
        self.window = int(window)        # > 0: sliding-window attention over the newest positions
        # > 0: every row's first shared_prefix_len cached tokens are the same
        # blocks (one prefill cloned N ways); attention reads them once per row group
        self.shared_prefix_len = int(shared_prefix_len)
        if self.shared_prefix_len and self.window:
            raise ValueError("a shared prefix and a sliding window do not combine")
        dt = k_cache.dtype
        # Per-step inputs and outputs live in two byte arenas (256-byte aligned
        # views), so a host-staged step moves each side with one copy.
        ins = [("q", (B, Hq, D), dt), ("k_new", (B, Hkv, D), dt), ("v_new", (B, Hkv, D), dt),
               ("block_tables", (B, max_blocks_per_seq), torch.int32), ("context_lens", (B,), torch.int32),
               ("temperature", (B,), torch.float32), ("top_k", (B,), torch.int32),
               ("top_p", (B,), torch.float32), ("seeds", (B,), torch.int64), ("offsets", (B,), torch.int64)]
        outs = [("out", (B, Hq, D), dt), ("token_ids", (B,), torch.int32)]
        # sampler extras: an allowed-id bit mask in, token_prob and the top-8 out
        self.extras = bool(extras)
        if self.extras:
            ins.append(("mask_words", (B, (vocab + 31) // 32), torch.int32))
            outs += [("token_prob", (B,), torch.float32), ("top_probs", (B, 8), torch.float32),
                     ("top_ids", (B, 8), torch.int32)]
        self._in_layout, in_bytes = _arena_layout(ins)
        self._out_layout, out_bytes = _arena_layout(outs)
        self.inputs = torch.zeros(in_bytes, dtype=torch.uint8, device=dev)
        self.outputs = torch.zeros(out_bytes, dtype=torch.uint8, device=dev)
        for name, view in _arena_views(self.inputs, self._in_layout).items():
            setattr(self, name, view)
        for name, view in _arena_views(self.outputs, self._out_layout).items():
            setattr(self, name, view)
        self.block_tables.fill_(-1)
        if self.extras:
            self.mask_words.fill_(-1)                  # every id allowed until the caller says otherwise
            n = ctypes.c_size_t(0)
            _capi.check(_capi.lib().pkvd_sample_workspace_bytes(B, vocab, ctypes.byref(n)))
            self.sample_workspace = torch.zeros(max(int(n.value), 16), dtype=torch.uint8, device=dev)
        self.temperature.fill_(1.0)
        self.top_p.fill_(1.0)
        self.slots = torch.empty(B, dtype=torch.int64, device=dev)
        self.logits = torch.zeros(B, vocab, dtype=logits_dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        nbytes = ctypes.c_size_t(0)
        if self.shared_prefix_len:
            _capi.check(_capi.lib().pkvd_decode_prefix_workspace_bytes(B, Hq, Hkv, D, max_context_len,
                                                                       self.shared_prefix_len, 0,
                                                                       ctypes.byref(nbytes)))
        else:
            _capi.check(_capi.lib().pkvd_decode_workspace_bytes(B, Hq, D, max_context_len, 0,
                                                                ctypes.byref(nbytes)))
        self.workspace = torch.zeros(max(int(nbytes.value), 16), dtype=torch.uint8, device=dev)
        self.cache = _capi.cache_desc(k_cache, v_cache)
        self.graph = None
        self.host_graph = None
        self.kernels_per_step = 5 if self.extras else 4   # store, partition, merge, sample (+ extras)

    def enqueue(self, stream=None) -> None:
        L = _capi.lib()
        s = _capi.stream_handle(stream, self.q)
        self._enqueue_kv_attention(L, s)
        self._enqueue_sample(L, s)

    def _enqueue_kv_attention(self, L, s) -> None:
        p = _capi.ptr
        # slot mapping and store in one kernel; the slots are kept for the caller
        _capi.check(L.pkvd_kv_store_paged(p(self.k_new), p(self.v_new), p(self.block_tables),
                                          self.block_tables.shape[1], p(self.context_lens), self.B,
                                          p(self.slots), ctypes.byref(self.cache), s, p(self.err)))
        self.enqueue_attention(L, s)

    def enqueue_attention(self, L=None, s=None) -> None:
        """The attention call of the step alone (on the current stream by default)."""
        L = L or _capi.lib()
        s = s if s is not None else _capi.stream_handle(None, self.q)
        p = _capi.ptr
        if self.shared_prefix_len:
            _capi.check(L.pkvd_paged_decode_attention_prefix(
                p(self.out), p(self.q), ctypes.byref(self.cache), p(self.block_tables),
                self.block_tables.shape[1], p(self.context_lens), self.max_context_len, self.B, self.Hq,
                ctypes.c_float(self.scale), self.shared_prefix_len, p(self.workspace), self.workspace.numel(), s,
                p(self.err)))
            return
        _capi.check(L.pkvd_paged_decode_attention_window(
            p(self.out), p(self.q), ctypes.byref(self.cache), p(self.block_tables),
            self.block_tables.shape[1], p(self.context_lens), self.max_context_len, self.B, self.Hq,
            ctypes.c_float(self.scale), self.window, p(self.workspace), self.workspace.numel(), s,
            p(self.err), self.path))

    def _enqueue_sample(self, L, s) -> None:
        p = _capi.ptr
        V = self.logits.shape[1]
        if self.extras:
            _capi.check(L.pkvd_sample_ex(p(self.token_ids), p(self.logits), _capi.dtype_code(self.logits.dtype),
                                         self.B, V, self.logits.stride(0), p(self.temperature), p(self.top_k),
                                         p(self.top_p), p(self.seeds), p(self.offsets), p(self.mask_words),
                                         self.mask_words.shape[1], p(self.token_prob), p(self.top_probs),
                                         p(self.top_ids), p(self.sample_workspace), self.sample_workspace.numel(), s))
            return
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

    # ------------------------------------------------ host-staged steps
    def host_buffers(self) -> dict:
        """Pinned host tensors shaped like the step's inputs and outputs
        (views of pinned arenas with the device arenas' layout), plus the
        logits: fill the inputs, call replay_host(), read out / token_ids."""
        if getattr(self, "_host", None) is None:
            hin = torch.zeros(self.inputs.numel(), dtype=torch.uint8, pin_memory=True)
            hout = torch.zeros(self.outputs.numel(), dtype=torch.uint8, pin_memory=True)
            h = {"_in": hin, "_out": hout,
                 "logits": torch.zeros(self.logits.shape, dtype=self.logits.dtype, pin_memory=True)}
            h.update(_arena_views(hin, self._in_layout))
            h.update(_arena_views(hout, self._out_layout))
            self._host = h
        return self._host

    def _enqueue_host(self) -> None:
        h = self.host_buffers()
        cur = torch.cuda.current_stream(self.q.device)
        self.inputs.copy_(h["_in"], non_blocking=True)
        # the logits are read by the sampler only: their copy runs on a
        # second stream, beside the store and attention kernels
        side = self._side
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            self.logits.copy_(h["logits"], non_blocking=True)
        L = _capi.lib()
        s = _capi.stream_handle(None, self.q)
        self._enqueue_kv_attention(L, s)
        # the attention output goes back to the host on a third stream,
        # beside the sampler (which does not touch it); the sampler's
        # outputs follow on this stream, which then joins the third
        out_side = self._side2
        out_side.wait_stream(cur)
        n_out = self._out_bytes("out")
        with torch.cuda.stream(out_side):
            h["_out"][:n_out].copy_(self.outputs[:n_out], non_blocking=True)
        cur.wait_stream(side)
        self._enqueue_sample(L, s)
        h["_out"][n_out:].copy_(self.outputs[n_out:], non_blocking=True)
        cur.wait_stream(out_side)

    def _out_bytes(self, name: str) -> int:
        """End offset of output `name` in the output arena (the first field
        starts at 0, so this is where the fields after it begin)."""
        for n, _shape, _dtype, off, nbytes in self._out_layout:
            if n == name:
                return off + (nbytes + 255) // 256 * 256
        raise KeyError(name)

    def capture_host(self) -> None:
        """Record a host-staged step (one input copy, the logits copy on a
        second stream, the kernels, the attention output's copy on a third
        stream beside the sampler, then the sampler's outputs) into a CUDA
        graph."""
        self._side = torch.cuda.Stream(device=self.q.device)
        self._side2 = torch.cuda.Stream(device=self.q.device)
        warm = torch.cuda.Stream(device=self.q.device)
        warm.wait_stream(torch.cuda.current_stream(self.q.device))
        with torch.cuda.stream(warm):
            self._enqueue_host()
        torch.cuda.current_stream(self.q.device).wait_stream(warm)
        torch.cuda.synchronize(self.q.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._enqueue_host()
        self.host_graph = g

    def replay_host(self) -> None:
        """One host-staged step; the host outputs are valid once the
        current stream has synchronised."""
        if self.host_graph is None:
            self.capture_host()
        self.host_graph.replay()


def _arena_layout(fields):
    layout, off = [], 0
    for name, shape, dtype in fields:
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        layout.append((name, shape, dtype, off, nbytes))
        off += (nbytes + 255) // 256 * 256
    return layout, max(off, 256)


def _arena_views(arena: torch.Tensor, layout) -> dict:
    return {name: arena[off:off + nbytes].view(dtype).view(shape) for name, shape, dtype, off, nbytes in layout}
