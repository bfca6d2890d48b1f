"""The benchmark's host-side oracle timing (the cpu_baseline and the
reference arm) on CPU: whole rows of a workload run in single-threaded
oracle processes, one pass on one process or cycling on several, and the
reference arm prints one JSON line with the contract's keys.  No GPU."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _tiny():
    import workloads
    from workloads import configs
    cfg = configs.get("tiny")
    return cfg, workloads.make_workload(cfg, device="cpu")


def test_single_process_does_one_pass_over_every_row():
    import bench
    cfg, w = _tiny()
    smp = bench.OracleSample(cfg, w)
    try:
        r = smp.run(30.0, procs=1)
    finally:
        smp.close()
    assert not os.path.exists(smp.path)
    assert r["rows"] == w.layout.num_seqs                # every row once, well inside the budget
    assert r["seconds"] >= r["attention_seconds"] > 0
    # the bytes of one pass over all rows are the workload's step and attention bytes
    b = bench.algorithmic_bytes(cfg, w.layout)
    assert r["bytes"] == b["step"] and r["attention_bytes"] == b["attention"]


def test_processes_share_the_rows_and_cycle_for_the_budget():
    import bench
    cfg, w = _tiny()
    smp = bench.OracleSample(cfg, w)
    try:
        r = smp.run(0.3, procs=3)
    finally:
        smp.close()
    done, secs, nbytes = r["rows"], r["seconds"], r["bytes"]
    assert r["procs"] == 3
    per_row = [bench.algorithmic_bytes(cfg, type(w.layout)(w.layout.context_lens[i:i + 1],
                                                           w.layout.block_tables[i:i + 1], w.layout.num_blocks,
                                                           w.layout.layer, w.layout.max_context_len))["step"]
               for i in range(w.layout.num_seqs)]
    assert done > w.layout.num_seqs                      # the rows were cycled
    assert 0.3 <= secs < 5.0
    assert min(per_row) * done <= nbytes <= max(per_row) * done


def test_reference_arm_prints_the_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "3", "--cpu-seconds", "1"], capture_output=True, text=True,
                       env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 1
    for key in ("metric", "value", "unit", "n_gpus", "ms_per_step", "higher_is_better", "config", "cpu_baseline",
                "e2e"):
        assert key in line, key
    # one single-threaded process per host core, at most one per row (tiny has 4 rows)
    assert line["cpu_baseline"]["cores"] == min(max(1, os.cpu_count() or 1), 4)
    assert line["cpu_baseline"]["value"] == line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and np.isfinite(line["e2e"]["value"])


def test_oracle_sample_keeps_mid_length_rows_within_its_byte_bound():
    """A long-context workload is sampled by whole mid-length rows under the
    float64 byte bound (the full workload would be tens of GB of float64)."""
    import bench
    import workloads
    from workloads import configs
    cfg = configs.LONGCTX.scaled(num_seqs=40, vocab=1000)
    w = workloads.make_workload(cfg, device="cpu")
    per_token = 2 * cfg.num_kv_heads * cfg.head_dim * 8
    smp = bench.OracleSample(cfg, w, max_bytes=200e6)
    try:
        ctx = w.layout.context_lens[smp.sel].astype(np.int64)
        assert 1 <= smp.num_rows < 40
        assert ctx.sum() * per_token <= 200e6 or smp.num_rows == 1
        med = np.median(w.layout.context_lens)
        assert ctx.max() <= np.max(w.layout.context_lens) and abs(np.median(ctx) - med) < med
    finally:
        smp.close()
