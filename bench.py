"""Benchmark of one paged-KV decode step on GB300.

A step is the whole hot path for one layer of one decode batch:
slot mapping -> KV store -> paged decode attention (partition + LSE merge)
-> fused sampler, replayed as one CUDA graph.  Inputs are seeded synthetic
tensors with the named workload's shapes, resident in HBM when timing
starts; L2 is flushed before every timed step or call, outside the timed
events (a 512 MB write, then a 512 MB read so the timed kernels find clean
lines).  The headline workload is the long-context batch (256 rows, 8.3 GB
of K/V per step); grok1, qwen3 and nanochat are timed in the same run under
`per_config`.

Reported (one JSON line on rank 0):
  value        decode-attention HBM GB/s: the attention's algorithmic bytes
               over the median of 100 timings of the attention call alone
               (partition + merge); ms_per_step and tokens_per_s are the whole
               step over the --steps timed steps, `step` its median and its
               fraction of the roofline
  roofline     the attention call against the measured HBM copy peak, with
               the DRAM traffic recorded by ncu for the current kernel sources
  attention_back_to_back, sampler
               the attention calls back to back (K/V larger than L2), and the
               sampler call alone
  e2e          the attention bytes over the step through the public API with
               host buffers: pinned host -> device copy of the step's inputs,
               the step, device -> host copy of its outputs, all timed
  cpu_baseline the float64 oracle on whole mid-length rows, on every host
               core (single-threaded processes), with the one-thread figure
  per_config   the same figures for the other workloads

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--per-config LIST|none]
    python bench.py --impl reference ...   (the oracle as the reference arm)
    python bench.py --profile-attention NAME --steps 3   (the command the DRAM captures profile)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402
from workloads import configs  # noqa: E402

METRIC = "decode-attention HBM GB/s (% of ~8 TB/s) and decode tokens/s per batch×ctx"
DEFAULT_CONFIG = "longctx"
FLUSH_BYTES = 512 << 20


class L2Flush:
    """Leaves L2 holding clean, unrelated lines: write a buffer larger than L2,
    then read a second one (so the timed kernel never pays for write-backs)."""

    def __init__(self, device):
        self.wbuf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.rbuf = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def add_(self, _):
        self.wbuf.add_(1)
        torch.sum(self.rbuf, dim=0, out=self.sink)


# ----------------------------------------------------------------- bytes
def algorithmic_bytes(cfg, layout, window=0, extras=False):
    """Bytes the method must move per step (each unique byte once); with a
    sliding window each row reads min(ctx, window) K/V rows."""
    s = cfg.itemsize
    B, Hq, Hkv, D, bs = layout.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.block_size
    ctx = layout.context_lens.astype(np.int64)
    nblk = -(-ctx // bs)
    if window > 0:
        start = np.maximum(ctx - window, 0)
        kv_tokens = int(np.sum(ctx - start))
        nblk = -(-ctx // bs) - start // bs          # table entries of the blocks the window touches
    elif cfg.table_kind == "shared_prefix":
        prefix = cfg.ctx_args[0]
        kv_tokens = prefix + int(np.sum(ctx - prefix))
    else:
        kv_tokens = int(ctx.sum())
    attn = kv_tokens * 2 * Hkv * D * s + 2 * B * Hq * D * s + int(nblk.sum()) * 4 + 4 * B
    store = 4 * B * Hkv * D * s + 8 * B
    slots = B * (4 + 4 + 8)
    sample = B * cfg.vocab * cfg.logits_itemsize + B * (4 + 4 + 4 + 8 + 8 + 4)
    if extras:                                      # mask bits in; token_prob and the top-8 out
        sample += B * ((cfg.vocab + 31) // 32) * 4 + B * (4 + 8 * 4 + 8 * 4)
    return {"attention": attn, "kv_store": store, "slot_mapping": slots, "sampler": sample,
            "step": attn + store + slots + sample}


def kernel_source_hash(prefix="attention"):
    """Hash of the kernel sources whose names start with `prefix`."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_kv_decode_store_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.startswith(prefix):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config_name, algorithmic, summary="attention_traffic.txt", prefix="attention"):
    """DRAM bytes (read + write) of one kernel launch from a committed ncu
    summary, if it was taken on the current kernel sources: {"bytes",
    "source"}, or None.  A record taken on a smaller profiling variant of the
    workload (the fourth field gives that variant's algorithmic bytes) is
    scaled to the full launch by the ratio of algorithmic bytes."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(prefix)
    for ln in open(path):
        parts = ln.split()
        if len(parts) >= 3 and not ln.startswith("#") and parts[0] == want and parts[1] == config_name:
            measured = int(parts[2])
            profiled = int(parts[3]) if len(parts) >= 4 and parts[3].isdigit() else algorithmic
            if profiled == algorithmic:
                return {"bytes": measured, "source": f"ncu, one launch of this workload ({summary})"}
            return {"bytes": int(round(measured * algorithmic / profiled)),
                    "source": f"ncu, one launch of a smaller variant ({profiled} algorithmic bytes, "
                              f"{measured} DRAM bytes), scaled by algorithmic bytes ({summary})"}
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = tempfile.mktemp(suffix=".csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in open(self.path):
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [x for x in sm if x >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- setup
def shared_prefix_of(lay, block_size):
    """Tokens every row of a batch shares (nanochat's cloned prefill), found
    from the host block tables as a scheduler would; 0 when none."""
    from paged_kv_decode_store_gb300 import shared_prefix_len
    return shared_prefix_len(lay.block_tables, lay.context_lens, block_size)


def build_step(cfg, device, path, window=0, extras=False, shared_prefix=None):
    import paged_kv_decode_store_gb300 as pk
    w = workloads.make_workload(cfg, device=device)
    lay = w.layout
    kc, vc = w.cache[0, lay.layer], w.cache[1, lay.layer]
    if shared_prefix is None:
        shared_prefix = 0 if window else shared_prefix_of(lay, cfg.block_size)
    step = pk.DecodeStep(kc, vc, lay.num_seqs, cfg.num_q_heads, lay.max_blocks_per_seq, lay.max_context_len,
                         cfg.vocab, w.logits.dtype, w.scale, path=path, window=window, extras=extras,
                         shared_prefix_len=shared_prefix)
    host = {
        "q": w.q, "k_new": w.k_new, "v_new": w.v_new,
        "block_tables": torch.from_numpy(lay.block_tables).to(device),
        "context_lens": torch.from_numpy(lay.context_lens).to(device),
        "logits": w.logits,
        "temperature": torch.from_numpy(w.temperature).to(device),
        "top_k": torch.from_numpy(w.top_k).to(device),
        "top_p": torch.from_numpy(w.top_p).to(device),
        "seeds": torch.from_numpy(w.seeds.view(np.int64)).to(device),
        "offsets": torch.from_numpy(w.offsets.view(np.int64)).to(device),
    }
    if extras:
        # a seeded 5 % of the vocabulary masked in every row
        g = torch.Generator(device="cpu").manual_seed(4242)
        allowed = torch.rand(lay.num_seqs, cfg.vocab, generator=g) >= 0.05
        host["mask_words"] = pk.pack_mask(allowed).to(device)
    for k, v in host.items():
        getattr(step, k).copy_(v)
    return w, step, host


def time_steps(step, flush, steps, stream):
    """Per-step CUDA-event durations (ms) of graph replays, L2 flushed before each."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.add_(1)
        starts[i].record(stream)
        step.replay()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_attention(step, flush, steps, stream):
    """Per-call CUDA-event durations (ms) of the attention call alone, replayed
    from its own CUDA graph right behind the L2 flush (no host gap inside)."""
    import paged_kv_decode_store_gb300 as pk

    def call():
        step.enqueue_attention()

    g = getattr(step, "_attn_graph", None)
    if g is None:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        step._attn_graph = g
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.add_(1)
        starts[i].record(stream)
        g.replay()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_attention_loop(step, calls, stream):
    """Mean per-call time (ms) of `calls` attention-graph replays back to back,
    between two CUDA events: the steady state of a layer loop, each call
    streaming its K/V from DRAM (only used where the K/V is larger than L2)."""
    time_attention(step, L2FlushNone(), 1, stream)          # makes sure the graph exists
    g = step._attn_graph
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(calls):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls


class L2FlushNone:
    def add_(self, _):
        pass


def time_sampler(step, flush, steps, stream):
    """Per-call CUDA-event durations (ms) of the sampler alone, replayed from
    its own CUDA graph right behind the L2 flush (the logits come from DRAM)."""
    import paged_kv_decode_store_gb300 as pk

    def call():
        step._enqueue_sample(pk.lib(), pk.stream_handle(None, step.q))

    g = getattr(step, "_samp_graph", None)
    if g is None:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        step._samp_graph = g
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.add_(1)
        starts[i].record(stream)
        g.replay()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_e2e(step, host_inputs, flush, steps, stream):
    """Public-API step with host buffers: one graph holds the H2D copy of the
    step's inputs (pinned arena), the logits' H2D copy on a second stream
    beside the store and attention kernels (which do not read them), the
    kernels, and the D2H copy of out and token ids."""
    h = step.host_buffers()
    for k, t in host_inputs.items():
        h[k].copy_(t)
    step.capture_host()
    h2d = h["_in"].numel() + h["logits"].numel() * h["logits"].element_size()
    d2h = h["_out"].numel()
    times = []
    for i in range(steps):
        flush.add_(1)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step.replay_host()
        torch.cuda.current_stream().synchronize()
        times.append((time.perf_counter() - t0) * 1e3)
    return times, h2d, d2h, h


# ----------------------------------------------------------------- oracle arm
ORACLE_SCRIPT = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
import oracle
d = np.load(sys.argv[2])
# the per-row inputs, read once (each access of an npz member reads it again)
q, knew, vnew, logits, ctx_all = d["q"], d["knew"], d["vnew"], d["logits"], d["ctx"]
temp, topk, topp, seeds = d["temp"], d["topk"], d["topp"], d["seeds"]
bs, scale = int(d["bs"]), float(d["scale"])
budget = float(sys.argv[3])
offset, stride, cycle = int(sys.argv[4]), int(sys.argv[5]), int(sys.argv[6])
mine = list(range(offset, int(q.shape[0]), stride))
counts, held = {}, {}
elapsed = 0.0      # oracle time only: reading a row's arrays from the file is not timed
attn = 0.0         # of which the attention call
k = 0
while mine and (k < len(mine) or cycle):
    i = mine[k % len(mine)]
    k += 1
    if i in held:
        kc, vc, tab = held[i]
    else:
        kc, vc, tab = d["k%d" % i], d["v%d" % i], d["t%d" % i][None, :]
        if cycle:
            held[i] = (kc, vc, tab)
    ctx = ctx_all[i:i + 1]
    t0 = time.perf_counter()
    slots = oracle.paging.decode_slot_mapping(tab, ctx, bs)
    oracle.store.kv_store(knew[i:i + 1], vnew[i:i + 1], slots, kc, vc)
    t1 = time.perf_counter()
    oracle.attention.decode_attention(q[i:i + 1], kc, vc, tab, ctx, scale)
    t2 = time.perf_counter()
    oracle.sampler.sample_row(logits[i], float(temp[i]), int(topk[i]), float(topp[i]), int(seeds[i]), 0)
    elapsed += time.perf_counter() - t0
    attn += t2 - t1
    counts[i] = counts.get(i, 0) + 1
    if elapsed > budget:
        break
print(json.dumps({"counts": counts, "seconds": elapsed, "attention_seconds": attn}))
"""


class OracleSample:
    """Whole rows of a decode workload (mid-length rows first, at most
    `max_rows` and `max_bytes` of float64 K/V) written once to a temporary
    file for the float64 oracle, which runs in single-threaded subprocesses
    (OMP/BLAS threads 1)."""

    def __init__(self, cfg, w, max_rows=None, max_bytes=1.5e9):
        self.cfg, self.lay = cfg, w.layout
        lay = self.lay
        B = lay.num_seqs if max_rows is None else min(max_rows, lay.num_seqs)
        order = np.argsort(lay.context_lens)[::-1]
        order = np.concatenate([order[len(order) // 2:], order[:len(order) // 2]])  # mid-length rows first
        per_token = 2 * cfg.num_kv_heads * cfg.head_dim * 8          # float64 K and V of one token
        sel, total = [], 0
        for i in order:
            if len(sel) >= B:
                break
            b = int(lay.context_lens[i]) * per_token
            if sel and total + b > max_bytes:
                continue
            sel.append(int(i))
            total += b
        sel = np.array(sel, dtype=np.int64)
        self.sel = sel
        rows = torch.from_numpy(sel.copy()).to(w.q.device)
        arrays = {"bs": np.array(cfg.block_size), "scale": np.array(w.scale)}
        arrays["q"] = w.q[rows].double().cpu().numpy()
        arrays["knew"] = w.k_new[rows].double().cpu().numpy()
        arrays["vnew"] = w.v_new[rows].double().cpu().numpy()
        arrays["logits"] = w.logits[rows].double().cpu().numpy()
        arrays["ctx"] = lay.context_lens[sel]
        arrays["temp"], arrays["topk"], arrays["topp"] = w.temperature[sel], w.top_k[sel], w.top_p[sel]
        arrays["seeds"] = w.seeds[sel]
        bs = cfg.block_size
        for j, i in enumerate(sel):
            n = -(-int(lay.context_lens[i]) // bs)
            idx = torch.from_numpy(lay.block_tables[i, :n].astype(np.int64)).to(w.cache.device)
            arrays["k%d" % j] = w.cache[0, lay.layer].index_select(0, idx).double().cpu().numpy()
            arrays["v%d" % j] = w.cache[1, lay.layer].index_select(0, idx).double().cpu().numpy()
            arrays["t%d" % j] = np.arange(n, dtype=np.int64)
        fd, self.path = tempfile.mkstemp(suffix=".npz")
        os.close(fd)
        np.savez(self.path, **arrays)
        self.row_bytes = {}

    @property
    def num_rows(self):
        return int(self.sel.shape[0])

    def bytes_of(self, i):
        """(step bytes, attention bytes) of row i alone."""
        if i not in self.row_bytes:
            lay = self.lay
            one = workloads.Layout(lay.context_lens[i:i + 1], lay.block_tables[i:i + 1], lay.num_blocks, lay.layer,
                                   lay.max_context_len)
            b = algorithmic_bytes(self.cfg, one)
            self.row_bytes[i] = (b["step"], b["attention"])
        return self.row_bytes[i]

    def run(self, budget_s, procs=1):
        """One bounded oracle run: {"rows", "seconds", "bytes", "attention_seconds",
        "attention_bytes", "procs"}.  procs == 1: one pass over the rows until
        ~budget_s of oracle time.  procs > 1: that many processes (at most one
        per row), started together, each cycling through its share of the rows
        for ~budget_s; the seconds are the slowest process's."""
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        procs = max(1, min(procs, self.num_rows))
        cycle = 1 if procs > 1 else 0
        ps = [subprocess.Popen([sys.executable, "-c", ORACLE_SCRIPT, ROOT, self.path, str(budget_s), str(k),
                                str(procs), str(cycle)], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                               env=env)
              for k in range(procs)]
        outs = [p.communicate() for p in ps]
        res = {"rows": 0, "seconds": 0.0, "bytes": 0, "attention_seconds": 0.0, "attention_bytes": 0,
               "procs": procs}
        for p, (out, err) in zip(ps, outs):
            if p.returncode:
                raise RuntimeError(err[-2000:])
            r = json.loads(out.strip().splitlines()[-1])
            res["seconds"] = max(res["seconds"], r["seconds"])
            res["attention_seconds"] = max(res["attention_seconds"], r["attention_seconds"])
            for j, c in r["counts"].items():
                sb, ab = self.bytes_of(int(self.sel[int(j)]))
                res["rows"] += c
                res["bytes"] += c * sb
                res["attention_bytes"] += c * ab
        return res

    def close(self):
        if os.path.exists(self.path):
            os.unlink(self.path)


def host_cores():
    return max(1, os.cpu_count() or 1)


def oracle_sample(cfg, w, budget_s=15.0, max_rows=None, procs=1):
    """One bounded oracle run on rows of the workload (see OracleSample.run)."""
    smp = OracleSample(cfg, w, max_rows)
    try:
        return smp.run(budget_s, procs)
    finally:
        smp.close()


# ----------------------------------------------------------------- main
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, cfg, ws, rank, local):
    """The oracle, as it stands, as the reference arm (rank 0 only): `value`
    is the same quantity as the GPU arm's, the attention's algorithmic bytes
    over the oracle's attention time."""
    if rank != 0:
        return
    w = workloads.make_workload(cfg, device=f"cuda:{local}" if torch.cuda.is_available() else "cpu")
    cores = host_cores()
    # a step: every host core runs the oracle on its share of the rows for a
    # bounded time, so the whole run stays within about a minute of oracle time
    budget = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps)))
    smp = OracleSample(cfg, w)
    tot = {"rows": 0, "seconds": 0.0, "bytes": 0, "attention_seconds": 0.0, "attention_bytes": 0}
    try:
        for _ in range(args.warmup):
            smp.run(min(1.0, budget), procs=cores)
        for _ in range(args.steps):
            r = smp.run(budget, procs=cores)
            procs = r["procs"]
            for key in tot:
                tot[key] += r[key]
    finally:
        smp.close()
    value = tot["attention_bytes"] / tot["attention_seconds"] / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot["seconds"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_block(cfg, w.layout),
            "tokens_per_s": tot["rows"] / tot["seconds"],
            "step_gbs": tot["bytes"] / tot["seconds"] / 1e9,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": procs, "kind": "oracle",
                             "sample": f"{tot['rows']} whole rows (store + attention + sampler; value = attention "
                                       f"bytes / attention time) of {smp.num_rows} mid-length rows, over "
                                       f"{args.steps} steps of ~{budget:.0f} s on {procs} single-threaded "
                                       f"processes (os.cpu_count() = {os.cpu_count()})"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_block(cfg, lay, window=0, extras=False):
    ctx = lay.context_lens
    desc = cfg.description + (f"; sliding window {window}" if window > 0 else "")
    desc += "; sampler extras (5% ids masked, token_prob, top-8)" if extras else ""
    return {"workload": desc, "name": cfg.name, "batch": int(lay.num_seqs),
            "ctx_mean": float(ctx.mean()), "ctx_max": int(ctx.max()), "q_heads": cfg.num_q_heads,
            "kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim, "block_size": cfg.block_size,
            "vocab": cfg.vocab,
            "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MB write, then {FLUSH_BYTES >> 20} MB read)"}


def device_l2_bytes():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size


def peak_hbm():
    """(HBM copy peak in GB/s, "measured" or "fallback")."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(path)).get("hbm_gbs") if os.path.exists(path) else None
    return (peak, "measured") if peak else (6800.0, "fallback")


def run_block_manager_bench(args):
    """The nanochat clone scenario on the host block manager (a 1024-token
    prompt, 16 forks, 255 decode appends each with copy-on-write on the first,
    release), timed through the Python binding, and the copy-on-write kernel
    moving whole blocks on the GPU."""
    import paged_kv_decode_store_gb300 as pk
    bs, nclone, ndec = 16, 16, 255
    rng = np.random.default_rng(7)
    prompt = rng.integers(0, 65536, 1024 + 7).tolist()          # 64 full blocks + a partial one
    t_alloc, t_fork, t_app, t_rel, n_app, copies = [], [], [], [], 0, 0
    for _ in range(max(args.steps, 3)):
        bm = pk.BlockManager(4096, bs)
        t0 = time.perf_counter()
        table, _ = bm.allocate(prompt)
        t_alloc.append(time.perf_counter() - t0)
        seqs = []
        t0 = time.perf_counter()
        for _ in range(nclone):
            seqs.append(bm.fork(table))
        t_fork.append((time.perf_counter() - t0) / nclone)
        bufs = [np.zeros(len(prompt) + ndec, dtype=np.int32) for _ in range(nclone)]   # token buffers
        for b in bufs:
            b[:len(prompt)] = prompt
        t0 = time.perf_counter()
        for d in range(ndec):
            n = len(prompt) + d + 1
            for i in range(nclone):
                bufs[i][n - 1] = d
                seqs[i], cp = bm.append(bufs[i][:n], seqs[i])
                copies += cp is not None
                n_app += 1
        t_app.append(time.perf_counter() - t0)
        t0 = time.perf_counter()
        for tab in seqs:
            bm.release(tab)
        bm.release(table)
        t_rel.append((time.perf_counter() - t0) / (nclone + 1))
        bm.close()
    # the copy kernel: 4096 whole blocks of the nanochat cache shape (bf16, 8 heads x 128)
    dev = "cuda"
    nb = 8192
    kc = torch.zeros(nb, bs, 8, 128, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    n = 4096
    src = torch.arange(n, dtype=torch.int32, device=dev)
    dst = src + n
    rows = torch.full((n,), bs, dtype=torch.int32, device=dev)
    for _ in range(3):
        pk.copy_blocks(kc, vc, src, dst, rows)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        pk.copy_blocks(kc, vc, src, dst, rows)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 10
    moved = 2 * n * 2 * kc[0].numel() * kc.element_size()       # K and V, read + write
    line = {"metric": "block manager op rates (host) and copy-on-write bandwidth (GPU)",
            "scenario": f"1031-token prompt, {nclone} forks, {ndec} appends each, block_size {bs}, 4096 blocks",
            "host_us": {"allocate": 1e6 * statistics.median(t_alloc), "fork": 1e6 * statistics.median(t_fork),
                        "append": 1e6 * sum(t_app) / n_app, "release": 1e6 * statistics.median(t_rel)},
            "copy_on_write_copies": copies, "timing": "through the Python binding (ctypes)",
            "copy_blocks": {"blocks": n, "ms": ms, "GB/s": moved / (ms * 1e-3) / 1e9,
                            "frac_of_copy_peak": moved / (ms * 1e-3) / 1e9 / peak_hbm()[0]}}
    print(json.dumps(line))


# ----------------------------------------------------------------- prefill
PREFILL_METRIC = "varlen paged prefill attention TFLOP/s (causal, prefix-cache hits)"

PREFILL_ORACLE_SCRIPT = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
import oracle
d = np.load(sys.argv[2])
budget = float(sys.argv[3])
cu_q, cu_k, tab, bs = d["cu_q"], d["cu_k"], d["tab"], int(d["bs"])
kc, vc = d["kc"], d["vc"]
slots = oracle.prefill.prefill_slot_mapping(tab, cu_q, cu_k, bs)
oracle.store.kv_store(d["knew"], d["vnew"], slots, kc, vc)
pairs = [tuple(int(x) for x in p) for p in d["pairs"]]
q, scale = d["q"], float(d["scale"])     # read once: each access of an npz member reads it again
t0 = time.perf_counter()
done = 0
while done < len(pairs) and time.perf_counter() - t0 < budget:
    oracle.prefill.prefill_attention(q, kc, vc, tab, cu_q, cu_k, scale, pairs=pairs[done:done + 16])
    done = min(done + 16, len(pairs))
print(json.dumps({"pairs": done, "seconds": time.perf_counter() - t0}))
"""


def prefill_keys(cu_q, cu_k, window=0):
    """Keys each new token attends to (causal, optional window), int64 [total_q]."""
    out = []
    for i in range(len(cu_q) - 1):
        qn, kn = int(cu_q[i + 1] - cu_q[i]), int(cu_k[i + 1] - cu_k[i])
        p = np.arange(kn - qn, kn, dtype=np.int64)
        first = np.maximum(p + 1 - window, 0) if window > 0 else np.zeros_like(p)
        out.append(p + 1 - first)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def prefill_oracle_sample(b, budget_s):
    """The float64 oracle on random (token, head) pairs of the median-length
    sequence, single-threaded, ~budget_s: (pairs done, seconds, FLOPs)."""
    klen = b.k_lens
    i = int(np.argsort(klen)[len(klen) // 2])
    bs, D = b.cfg.block_size, b.cfg.head_dim
    n = -(-int(klen[i]) // bs)
    ids = torch.from_numpy(b.block_tables[i, :n].astype(np.int64))
    q0, q1 = int(b.cu_seqlens_q[i]), int(b.cu_seqlens_q[i + 1])
    rng = np.random.default_rng(3)
    toks = rng.integers(0, q1 - q0, 4096)
    heads = rng.integers(0, b.cfg.num_q_heads, 4096)
    arrays = {"cu_q": np.array([0, q1 - q0]), "cu_k": np.array([0, int(klen[i])]),
              "tab": np.arange(n, dtype=np.int64)[None, :], "bs": np.array(bs), "scale": np.array(b.scale),
              "kc": b.cache[0].index_select(0, ids).double().numpy(),
              "vc": b.cache[1].index_select(0, ids).double().numpy(),
              "knew": b.k_new[q0:q1].double().numpy(), "vnew": b.v_new[q0:q1].double().numpy(),
              "q": b.q[q0:q1].double().numpy(), "pairs": np.stack([toks, heads], 1)}
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    np.savez(path, **arrays)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", PREFILL_ORACLE_SCRIPT, ROOT, path, str(budget_s)],
                       capture_output=True, text=True, env=env)
    os.unlink(path)
    if r.returncode:
        raise RuntimeError(r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    keys = prefill_keys(arrays["cu_q"], arrays["cu_k"])
    flops = 4.0 * D * float(keys[toks[:res["pairs"]]].sum())
    return res["pairs"], res["seconds"], flops


def run_prefill_bench(args):
    """One prefill step (varlen store + causal attention over the paged cache)
    of a seeded batch, replayed as a CUDA graph, L2 flushed before each step."""
    import paged_kv_decode_store_gb300 as pk
    from workloads import prefill as wp
    cfg = wp.PREFILL_CONFIGS[args.prefill]
    b = wp.make_prefill_batch(cfg)
    dev = "cuda:0"
    torch.cuda.set_device(0)
    window = args.window
    cache = b.cache.to(dev)
    kc, vc = cache[0], cache[1]
    d = {"q": b.q.to(dev), "k": b.k_new.to(dev), "v": b.v_new.to(dev),
         "tables": torch.from_numpy(b.block_tables).to(dev), "cu_q": torch.from_numpy(b.cu_seqlens_q).to(dev),
         "cu_k": torch.from_numpy(b.cu_seqlens_k).to(dev)}
    out = torch.empty_like(d["q"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    maxq = b.max_seqlen_q

    def store():
        pk.kv_store_prefill(d["k"], d["v"], d["tables"], d["cu_q"], d["cu_k"], kc, vc, err=err)

    path = {"auto": pk.PATH_AUTO, "tc": pk.PATH_TC, "mma": pk.PATH_MMA, "fma": pk.PATH_FMA}[args.prefill_path]

    def attend():
        pk.prefill_attention(d["q"], kc, vc, d["tables"], d["cu_q"], d["cu_k"], maxq, b.scale, window=window,
                             out=out, err=err, path=path)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        store()
        attend()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        store()
        attend()
    with torch.cuda.graph(g_attn):
        attend()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def timed(graph, n):
        st = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for j in range(n):
            flush.add_(1)
            st[j].record(stream)
            graph.replay()
            en[j].record(stream)
        torch.cuda.synchronize()
        return [x.elapsed_time(y) for x, y in zip(st, en)]

    timed(g_step, args.warmup)
    timed(g_attn, 3)
    with ClockSampler(0) as clk:
        step_ms = timed(g_step, args.steps)
        attn_ms = timed(g_attn, args.steps)
    clocks = clk.summary()

    # end to end: pinned host inputs -> device, the step, the output -> pinned host
    host_in = {k: t.cpu().pin_memory() for k, t in d.items()}
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    e2e = []
    for j in range(args.warmup + args.steps):
        flush.add_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k, t in host_in.items():
            d[k].copy_(t, non_blocking=True)
        g_step.replay()
        host_out.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if j >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    if int(err.item()):
        raise RuntimeError(f"prefill kernels flagged device errors {int(err.item())}")

    keys = prefill_keys(b.cu_seqlens_q, b.cu_seqlens_k, window)
    flops = 4.0 * cfg.num_q_heads * cfg.head_dim * float(keys.sum())
    ms = statistics.mean(step_ms)
    attn = statistics.mean(attn_ms)
    e2e_ms = statistics.mean(e2e)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = peaks.get("bf16_tflops") or 1900.0
    achieved = flops / (attn * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": cfg.description + (f"; sliding window {window}" if window else ""),
                   "name": cfg.name, "batch": cfg.num_seqs, "total_q": b.total_q,
                   "q_len_mean": float(b.q_lens.mean()), "cached_mean": float((b.k_lens - b.q_lens).mean()),
                   "max_seqlen_q": maxq, "q_heads": cfg.num_q_heads, "kv_heads": cfg.num_kv_heads,
                   "head_dim": cfg.head_dim, "block_size": cfg.block_size,
                   "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MB write, then "
                         f"{FLUSH_BYTES >> 20} MB read)"},
        "tokens_per_s": b.total_q / (ms * 1e-3), "attention_flops": flops, "attention_ms": attn,
        "attention_path": args.prefill_path,
        "roofline": {"kernel": ("prefill_attention_kernel (mma.sync m16n8k16, fp32 accumulation)"
                                if args.prefill_path == "mma" else
                                "prefill_fma_kernel (fp32 CUDA-core dot products)" if args.prefill_path == "fma" else
                                "prefill_tc_kernel (tcgen05.mma kind::f16, TMA 128B-swizzled K/V, TMEM accumulators)"),
                     "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "peak_source": "measured bf16 burst" if peaks.get("bf16_tflops") else "fallback",
                     "traffic": None if args.prefill_path in ("mma", "fma") else
                     (recorded_traffic(cfg.name, None, "prefill_traffic.txt", "prefill_tc") or {}).get("bytes")},
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps, "clocks": clocks, "device_err_flag": 0,
    }
    if not args.no_cpu_baseline:
        done, secs, cflops = prefill_oracle_sample(b, args.cpu_seconds)
        line["cpu_baseline"] = {"value": cflops / secs / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                "sample": f"{done} random (token, head) rows of the median sequence, "
                                          f"{secs:.1f} s, single thread"}
    print(json.dumps(line))


# ----------------------------------------------------------------- serving timeline
SERVE_DECODE_CONFIG = {"qwen3_prefill": "qwen3", "grok1_prefill": "grok1", "chunked_prefill": "longctx"}


def run_serve_bench(args):
    """One layer's hot path over a request's life: the prefill step of a batch
    (store + causal attention over the cached prefixes + first-token sample),
    then `steps` decode steps on the same paged cache (store + decode
    attention + sample, one CUDA graph each).  Reports TTFT, TPOT and tok/s
    (nanochat "04 · Engine", section "推理基准 infer_bench.py": TTFT / TPOT /
    tok/s, with MFU for the compute-bound prefill and MBU for the
    bandwidth-bound decode, and decode tok/s bounded by peak bandwidth over
    the bytes read per step)."""
    import paged_kv_decode_store_gb300 as pk
    from workloads import prefill as wp
    pcfg = wp.PREFILL_CONFIGS[args.serve]
    dcfg = configs.get(SERVE_DECODE_CONFIG[args.serve])
    b = wp.make_prefill_batch(pcfg)
    dev = "cuda:0"
    torch.cuda.set_device(0)
    B, bs, gen = pcfg.num_seqs, pcfg.block_size, max(args.steps, 4)
    Hq, Hkv, D = pcfg.num_q_heads, pcfg.num_kv_heads, pcfg.head_dim
    k_lens = b.k_lens.astype(np.int64)
    # tables with room for `gen` more tokens: new blocks appended after the pool
    need = [-(-int(k + gen) // bs) for k in k_lens]
    width = max(need)
    tables = np.full((B, width), -1, dtype=np.int32)
    nb = b.num_blocks
    for i in range(B):
        have = -(-int(k_lens[i]) // bs)
        tables[i, :have] = b.block_tables[i, :have]
        tables[i, have:need[i]] = np.arange(nb, nb + need[i] - have)
        nb += need[i] - have
    cache = torch.empty((2, nb) + tuple(b.cache.shape[2:]), dtype=b.cache.dtype, device=dev)
    cache[:, :b.num_blocks].copy_(b.cache.to(dev))
    cache[:, b.num_blocks:].normal_()
    kc, vc = cache[0], cache[1]
    d = {"q": b.q.to(dev), "k": b.k_new.to(dev), "v": b.v_new.to(dev),
         "tables": torch.from_numpy(tables).to(dev), "cu_q": torch.from_numpy(b.cu_seqlens_q).to(dev),
         "cu_k": torch.from_numpy(b.cu_seqlens_k).to(dev)}
    out = torch.empty_like(d["q"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(77)
    ldt = workloads.synth.TORCH_DTYPES[dcfg.logits_dtype]
    logits = torch.randn((B, dcfg.vocab), generator=g, device=dev).mul_(dcfg.logits_std).to(ldt)
    temp = torch.full((B,), 0.8, device=dev)
    top_k = torch.zeros(B, dtype=torch.int32, device=dev)
    top_p = torch.full((B,), 0.95, device=dev)
    seeds = torch.arange(B, dtype=torch.int64, device=dev) * 7919 + 1
    offs = torch.zeros(B, dtype=torch.int64, device=dev)
    first = torch.empty(B, dtype=torch.int32, device=dev)

    def prefill():
        pk.kv_store_prefill(d["k"], d["v"], d["tables"], d["cu_q"], d["cu_k"], kc, vc, err=err)
        pk.prefill_attention(d["q"], kc, vc, d["tables"], d["cu_q"], d["cu_k"], b.max_seqlen_q, b.scale, out=out,
                             err=err)
        pk.sample(logits, temp, top_k, top_p, seeds, offs, out=first)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        prefill()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g_pre = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pre):
        prefill()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    ttft = []
    for j in range(args.warmup + args.steps):
        flush.add_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g_pre.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if j >= args.warmup:
            ttft.append(e0.elapsed_time(e1))

    # decode: the token at position k_len (then k_len + 1, ...) of every sequence
    step = pk.DecodeStep(kc, vc, B, Hq, width, int(k_lens.max()) + gen, dcfg.vocab, ldt, b.scale)
    step.q.normal_(generator=g)
    step.k_new.normal_(generator=g)
    step.v_new.normal_(generator=g)
    step.block_tables.copy_(d["tables"])
    ctx0 = torch.from_numpy((k_lens + 1).astype(np.int32)).to(dev)
    step.context_lens.copy_(ctx0)
    step.logits.copy_(logits)
    step.temperature.copy_(temp)
    step.top_p.copy_(top_p)
    step.seeds.copy_(seeds)
    step.capture()
    tpot = []
    for rnd in range(2):                    # a warm-up pass over the timeline, then the timed one
        step.context_lens.copy_(ctx0)
        for t in range(gen):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step.replay()
            e1.record(stream)
            step.context_lens.add_(1)       # the scheduler's bookkeeping between steps
            step.offsets.add_(1)
            if rnd:
                tpot.append((e0, e1))
    torch.cuda.synchronize()
    tpot = [x.elapsed_time(y) for x, y in tpot]
    if int(err.item()) or int(step.err.item()):
        raise RuntimeError(f"device error flags {int(err.item())} / {int(step.err.item())}")

    keys = prefill_keys(b.cu_seqlens_q, b.cu_seqlens_k)
    flops = 4.0 * Hq * D * float(keys.sum())
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak_t = peaks.get("bf16_tflops") or 1900.0
    peak_b, _ = peak_hbm()
    dec_cfg = dcfg.scaled(num_seqs=B, table_kind="perm")
    mid_ctx = (k_lens + 1 + gen // 2).astype(np.int32)
    lay = workloads.Layout(mid_ctx, tables, nb, 0, int(mid_ctx.max()))
    step_bytes = algorithmic_bytes(dec_cfg, lay)["step"]
    ttft_ms, tpot_ms = statistics.mean(ttft), statistics.mean(tpot)
    line = {
        "metric": "serving timeline of one layer's hot path: TTFT, TPOT, tok/s; MFU (prefill), MBU (decode)",
        "value": B / (tpot_ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": gen, "warmup": args.warmup,
        "higher_is_better": True, "dtype": pcfg.dtype, "data": "synthetic",
        "config": {"workload": pcfg.description + f"; then {gen} decode steps on the same cache",
                   "prefill": pcfg.name, "decode_shapes": dcfg.name, "batch": B, "prompt_tokens": int(b.total_q),
                   "cached_tokens": int((k_lens - b.q_lens).sum()), "vocab": dcfg.vocab,
                   "l2": "flushed before each prefill; decode steps back to back (steady state)"},
        "ttft_ms": ttft_ms, "tpot_ms": tpot_ms, "tokens_per_s": B / (tpot_ms * 1e-3),
        "mfu_prefill": flops / (ttft_ms * 1e-3) / 1e12 / peak_t,
        "mbu_decode": step_bytes / (tpot_ms * 1e-3) / 1e9 / peak_b,
        "decode_step_bytes": step_bytes,
        "decode_tokens_per_s_bound": B * peak_b * 1e9 / step_bytes,
        "peaks": {"tflops": peak_t, "hbm_gbs": peak_b},
        "gpu_launches": 3 * len(ttft) + step.kernels_per_step * gen,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--path", default="auto", choices=["auto", "fma", "mma"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extras", action="store_true",
                    help="sampler extras: a 5 %% id mask, token_prob and the top-8 probabilities and ids")
    ap.add_argument("--block-manager", action="store_true",
                    help="host block manager op rates and the copy-on-write kernel's bandwidth (one JSON line)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window attention over the newest W positions (0: none)")
    ap.add_argument("--prefill", default=None,
                    choices=["qwen3_prefill", "grok1_prefill", "chunked_prefill"],
                    help="time a varlen prefill step (store + causal attention) instead (one JSON line)")
    ap.add_argument("--prefill-path", default="auto", choices=["auto", "tc", "mma", "fma"],
                    help="prefill attention kernel: tcgen05 (auto picks it where it runs), mma.sync or CUDA cores")
    ap.add_argument("--per-config", default="grok1,qwen3,nanochat",
                    help="more decode workloads timed after the headline one, in the same line (none: skip)")
    ap.add_argument("--profile-attention", default=None, choices=sorted(PROFILE_VARIANTS),
                    help="run one workload's attention call --steps times (the command ncu captures)")
    ap.add_argument("--serve", default=None, choices=["qwen3_prefill", "grok1_prefill", "chunked_prefill"],
                    help="serving timeline: the batch's prefill, then --steps decode steps (TTFT / TPOT, one line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = configs.get(args.config)
    ws, rank, local = dist_setup()

    if args.impl == "reference":
        run_reference(args, cfg, ws, rank, local)
        return
    if args.block_manager:
        if rank == 0:
            run_block_manager_bench(args)
        return
    if args.profile_attention:
        if rank == 0:
            run_profile_attention(args)
        return
    if args.prefill:
        if rank == 0:
            run_prefill_bench(args)
        return
    if args.serve:
        if rank == 0:
            run_serve_bench(args)
        return

    import paged_kv_decode_store_gb300 as pk
    path = {"auto": pk.PATH_AUTO, "fma": pk.PATH_FMA, "mma": pk.PATH_MMA}[args.path]
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    w, step, host = build_step(cfg, dev, path, window=args.window, extras=args.extras)
    lay = w.layout
    nbytes = algorithmic_bytes(cfg, lay, window=args.window, extras=args.extras)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    n_attn = max(args.steps, ATTENTION_TIMINGS)

    step.capture()
    for _ in range(args.warmup):
        flush.add_(1)
        step.replay()
    time_attention(step, flush, 3, stream)
    torch.cuda.synchronize()

    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_ms = time_steps(step, flush, args.steps, stream)
        torch.cuda.synchronize()
        barrier(ws)
        attn_ms = time_attention(step, flush, n_attn, stream)
    torch.cuda.synchronize()
    barrier(ws)
    total_ms = max_over_ranks(sum(step_ms), ws, dev)
    step_med = max_over_ranks(statistics.median(step_ms), ws, dev)
    attn_med = max_over_ranks(statistics.median(attn_ms), ws, dev)
    clocks = clk.summary()
    time_sampler(step, flush, 3, stream)
    samp_ms = time_sampler(step, flush, n_attn, stream)
    loop_ms = time_attention_loop(step, n_attn, stream) if nbytes["attention"] > device_l2_bytes() else None

    pinned = {k: v.cpu() for k, v in host.items()}
    for _ in range(2):
        time_e2e(step, pinned, flush, 1, stream)
    e2e_ms, h2d, d2h, hb = time_e2e(step, pinned, flush, args.steps, stream)
    if not torch.equal(hb["token_ids"], step.token_ids.cpu()):
        raise RuntimeError("host-staged step disagrees with the device step")
    e2e_total = max_over_ranks(sum(e2e_ms), ws, dev)
    err = int(step.err.item())

    if rank != 0:
        return
    ms_per_step = total_ms / args.steps
    peak, peak_src = peak_hbm()
    attn_gbs = nbytes["attention"] / (attn_med * 1e-3) / 1e9
    step_gbs = nbytes["step"] / (step_med * 1e-3) / 1e9
    traffic = recorded_traffic(cfg.name, nbytes["attention"]) if not args.window else None
    e2e_step_ms = e2e_total / args.steps
    line = {
        "metric": METRIC, "value": ws * attn_gbs, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": config_block(cfg, lay, args.window, args.extras),
        "value_is": (f"paged decode attention (partition + LSE merge) algorithmic HBM bytes / median attention "
                     f"time over {n_attn} graph replays, L2 flushed before each; ms_per_step and tokens_per_s "
                     f"are the whole step (store, attention, merge, sampler) over the {args.steps} timed steps"),
        "tokens_per_s": ws * lay.num_seqs / (ms_per_step * 1e-3),
        "step": {"ms_median": step_med, "ms_mean": ms_per_step, "bytes": nbytes["step"], "gbs": ws * step_gbs,
                 "frac": step_gbs / peak, "tokens_per_s_median": ws * lay.num_seqs / (step_med * 1e-3)},
        "attention_bytes": nbytes["attention"], "attention_ms_median": attn_med,
        "attention_ms_mean": statistics.mean(attn_ms), "attention_path": args.path,
        "attention_back_to_back": loop_ms and {
            "ms_per_call": loop_ms, "gbs": nbytes["attention"] / (loop_ms * 1e-3) / 1e9,
            "frac": nbytes["attention"] / (loop_ms * 1e-3) / 1e9 / peak,
            "is": f"{n_attn} attention calls back to back between two events (K/V larger than L2, so each "
                  "call streams from DRAM): the steady state of a loop over layers"},
        "sampler": {"ms_median": statistics.median(samp_ms), "bytes": nbytes["sampler"],
                    "gbs": nbytes["sampler"] / (statistics.median(samp_ms) * 1e-3) / 1e9,
                    "frac": nbytes["sampler"] / (statistics.median(samp_ms) * 1e-3) / 1e9 / peak,
                    "is": f"the sampler call alone, median of {n_attn} graph replays, L2 flushed before each"},
        "roofline": {"kernel": "paged_decode_attention (partition + LSE merge kernels)", "bound": "hbm",
                     "achieved": attn_gbs, "peak": peak, "unit": "GB/s", "frac": attn_gbs / peak,
                     "peak_source": f"{peak_src} (copy peak, burst)", "traffic": traffic and traffic["bytes"],
                     "traffic_source": traffic and traffic["source"]},
        "e2e": {"value": ws * nbytes["attention"] / (e2e_step_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_step_ms, "tokens_per_s": ws * lay.num_seqs / (e2e_step_ms * 1e-3),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "is": "the attention bytes over the whole host-staged step (inputs copied in from pinned memory, "
                      "the step, outputs copied back)"},
        # the step graph's kernels, plus partition + merge of the attention-only replays
        # (the sampler-alone and back-to-back timings run after the timed region)
        "gpu_launches": step.kernels_per_step * args.steps + 2 * n_attn,
        "clocks": clocks, "device_err_flag": err,
    }
    if not args.no_cpu_baseline and ws == 1:
        # the oracle on the host: one thread (one pass over the rows), then
        # every core (single-threaded processes over shares of the rows)
        cores = host_cores()
        smp = OracleSample(cfg, w)
        try:
            one = smp.run(args.cpu_seconds, procs=1)
            alln = smp.run(max(1.0, min(args.cpu_seconds, 30.0 / cores)), procs=cores)
        finally:
            smp.close()
        line["cpu_baseline"] = {
            "value": alln["attention_bytes"] / alln["attention_seconds"] / 1e9, "unit": "GB/s",
            "cores": alln["procs"], "kind": "oracle",
            "sample": f"{alln['rows']} whole rows (store + attention + sampler) of {smp.num_rows} mid-length rows "
                      f"of this workload in {alln['seconds']:.1f} s on {alln['procs']} single-threaded processes "
                      f"(os.cpu_count() = {os.cpu_count()}); value = attention bytes / attention time",
            "step_gbs": alln["bytes"] / alln["seconds"] / 1e9,
            "tokens_per_s": alln["rows"] / alln["seconds"],
            "single_thread": {"value": one["attention_bytes"] / one["attention_seconds"] / 1e9, "unit": "GB/s",
                              "cores": 1, "sample": f"{one['rows']} whole rows, {one['seconds']:.1f} s"}}
    others = [c for c in args.per_config.split(",") if c and c != "none" and c != cfg.name]
    if others and ws == 1:
        del w, step, host, pinned, hb
        torch.cuda.empty_cache()
        line["per_config"] = {name: measure_config(configs.get(name), dev, path, args, flush, stream, local,
                                                   peak)
                              for name in others}
    print(json.dumps(line))


ATTENTION_TIMINGS = 100           # attention-call timings per workload (the median is reported)


def measure_config(cfg, dev, path, args, flush, stream, local, peak):
    """One more workload, timed like the headline one (its own clock record):
    attention alone (median of ATTENTION_TIMINGS graph replays) and the whole
    step (median of as many replays), each against the HBM roofline."""
    w, step, host = build_step(cfg, dev, path)
    lay = w.layout
    nbytes = algorithmic_bytes(cfg, lay)
    n = max(args.steps, ATTENTION_TIMINGS)
    step.capture()
    for _ in range(args.warmup):
        flush.add_(1)
        step.replay()
    time_attention(step, flush, 3, stream)
    torch.cuda.synchronize()
    time_sampler(step, flush, 3, stream)
    with ClockSampler(local) as clk:
        step_ms = time_steps(step, flush, n, stream)
        attn_ms = time_attention(step, flush, n, stream)
        samp_ms = time_sampler(step, flush, n, stream)
    torch.cuda.synchronize()
    err = int(step.err.item())
    a_med, s_med = statistics.median(attn_ms), statistics.median(step_ms)
    sp_med = statistics.median(samp_ms)
    l2 = device_l2_bytes()
    loop_ms = time_attention_loop(step, n, stream) if nbytes["attention"] > l2 else None
    a_gbs = nbytes["attention"] / (a_med * 1e-3) / 1e9
    s_gbs = nbytes["step"] / (s_med * 1e-3) / 1e9
    traffic = recorded_traffic(cfg.name, nbytes["attention"])
    plain_us = None
    if step.shared_prefix_len:
        # the same call through the plain kernel, which reads the prefix once per row
        w2, step2, _ = build_step(cfg, dev, path, shared_prefix=0)
        step2.enqueue()
        time_attention(step2, flush, 3, stream)
        plain_us = 1e3 * statistics.median(time_attention(step2, flush, n, stream))
        del w2, step2
    res = {"workload": cfg.description, "timings": n,
           "attention_call": ("pkvd_paged_decode_attention_prefix (shared prefix of "
                              f"{step.shared_prefix_len} tokens)") if step.shared_prefix_len
                             else "pkvd_paged_decode_attention",
           "attention_plain_kernel_us": plain_us,
           "attention_us": 1e3 * a_med, "attention_bytes": nbytes["attention"], "attention_gbs": a_gbs,
           "attention_frac": a_gbs / peak,
           "traffic": traffic and traffic["bytes"], "traffic_source": traffic and traffic["source"],
           "traffic_over_algorithmic": traffic and traffic["bytes"] / nbytes["attention"],
           "attention_us_back_to_back": loop_ms and 1e3 * loop_ms,
           "attention_frac_back_to_back": loop_ms and nbytes["attention"] / (loop_ms * 1e-3) / 1e9 / peak,
           "sampler_us": 1e3 * sp_med, "sampler_bytes": nbytes["sampler"],
           "sampler_gbs": nbytes["sampler"] / (sp_med * 1e-3) / 1e9,
           "sampler_frac": nbytes["sampler"] / (sp_med * 1e-3) / 1e9 / peak,
           "step_us": 1e3 * s_med, "step_bytes": nbytes["step"], "step_gbs": s_gbs, "step_frac": s_gbs / peak,
           "tokens_per_s": lay.num_seqs / (s_med * 1e-3), "clocks": clk.summary(), "device_err_flag": err}
    del w, step, host
    torch.cuda.empty_cache()
    return res


def run_profile_attention(args):
    """The attention call of a workload (its profiling variant, small enough
    for counter captures), `--steps` times back to back after one store: the
    command that ncu captures for the DRAM-traffic records."""
    import paged_kv_decode_store_gb300 as pk
    cfg = PROFILE_VARIANTS[args.profile_attention]
    dev = "cuda:0"
    torch.cuda.set_device(0)
    w, step, _ = build_step(cfg, dev, pk.PATH_AUTO)
    step.enqueue()
    for _ in range(args.steps):
        step.enqueue_attention()          # the step's own attention call (shared-prefix where the rows share one)
    torch.cuda.synchronize()
    if int(step.err.item()):
        raise RuntimeError(f"device error flag {int(step.err.item())}")
    nbytes = algorithmic_bytes(cfg, w.layout)
    print(json.dumps({"profile_attention": args.profile_attention, "attention_bytes": nbytes["attention"],
                      "calls": args.steps, "workload": cfg.description, "num_seqs": cfg.num_seqs,
                      "num_layers": cfg.num_layers,
                      "device_gb": torch.cuda.max_memory_allocated() / 1e9}))


# Workloads whose attention launch ncu captures for DRAM traffic: the full
# shapes where the device footprint is small, else the same shapes with a
# smaller pool (one cache layer; a quarter of the rows).
PROFILE_VARIANTS = {
    "grok1": configs.GROK1,
    "nanochat": configs.NANOCHAT,
    "qwen3": configs.QWEN3.scaled(num_layers=1),
    "longctx": configs.LONGCTX.scaled(num_seqs=64),
}


if __name__ == "__main__":
    main()
