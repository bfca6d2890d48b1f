"""Plain float64 CPU oracle for the paged decode step.  TEST INFRASTRUCTURE ONLY.

This package is the independent reference the CUDA path is checked against.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it; the library and its Python binding never do, and it shares no
code, constants or helpers with them.

Every function restates, in the plainest form, what the pages define:

* ``paging``    -- slot arithmetic and cache sizing (nano-vllm "Model Runner",
  section "allocated kv cache"; Grok-1 "第 8 章 runners.py 推理引擎",
  section 8.5).
* ``store``     -- the scalar cache store through ``slot_mapping``.
* ``attention`` -- gather, softmax, weighted sum over a sequence's block
  table, in float64; plus the log-sum-exp merge of partial states.
* ``philox``    -- Philox4x32-10 from its published definition (Salmon,
  Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).
* ``sampler``   -- temperature, top-k, nucleus cut (Grok-1 section 8.3.1
  ``top_p_filter``, restated in descending order), Gumbel-max draw.
* ``prefill``   -- varlen prefill: slots of the scheduled tokens and causal
  attention over cached prefix plus new rows (nano-vllm "Model Runner",
  sections "prefix cache", "prepare Prefill", "prefill and decode").
* ``block_manager`` -- block allocation with prefix sharing, forks and
  copy-on-write (imported on its own by its tests).

Pins: every function is checked by ``tests/test_oracle_*.py`` against
worked examples the pages print, closed forms, brute force on tiny inputs,
library routines and published known-answer vectors.  No function is left
"parity unpinned".
"""
from . import paging, store, attention, philox, sampler, prefill  # noqa: F401
