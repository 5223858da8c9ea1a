"""Seeded synthetic inputs for the dual-flow decode step.

This package is shared by the CPU oracle's tests, the CUDA-path tests and the
benchmark.  It holds workload descriptions (sizes only) and counter-based
generators for weights, token ids and synthetic KV-cache contents.  It holds
none of the method's arithmetic: nothing here normalises, projects, attends,
mixes or routes.
"""

from .configs import DFConfig, WORKLOADS, TEST_CONFIGS, get_config  # noqa: F401
from .gen import (  # noqa: F401
    Weights,
    DeviceWeights,
    tokens,
    prompt_lengths,
    synthetic_kv_block,
    bf16_round_f32,
    tensor_id,
)
