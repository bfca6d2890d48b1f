"""Seeded synthetic decode-step workloads (inputs only, no decode arithmetic)."""
from .configs import CONFIGS, BY_INDEX, DecodeConfig, get  # noqa: F401
from .synth import (Layout, SamplerInputs, Workload, make_layout, make_sampler_inputs,  # noqa: F401
                    make_workload, poison_rows)
