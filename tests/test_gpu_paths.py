"""The tensor-core / TMA fast paths against the CUDA-core path of the same
library on identical inputs.  Both compute the same quantities with fp32
accumulation, so they agree to accumulation-order rounding; this isolates a
fault in a fast kernel from the oracle comparison."""

import os

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights

from parity_util import GpuRun

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["t_bf16", "t_bf16_b9", "t_moe"])
def test_fast_path_matches_cuda_core_path(name, cuda_device):
    cfg = dfsynth.get_config(name).with_(n_steps=3)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    os.environ["DF_FORCE_GENERIC"] = "1"
    try:
        ref = GpuRun(cfg, w, tok)
    finally:
        del os.environ["DF_FORCE_GENERIC"]
    fast = GpuRun(cfg, w, tok)
    for a, b in zip(fast.steps, ref.steps):
        d1 = np.abs(a["logp1"] - b["logp1"]).max()
        dm = np.abs(a["logp_mix"] - b["logp_mix"]).max()
        print(name, "max |dlogp1|", d1, "max |dlogp_mix|", dm)
        assert d1 < 5e-3 and dm < 5e-3
    diff = np.abs(fast.kv - ref.kv).astype(np.float64)
    rel = float(np.sqrt((diff ** 2).sum() / (ref.kv.astype(np.float64) ** 2).sum()))
    print("kv max", diff.max(), "relative rms", rel)
    assert diff.max() < 0.05 and rel < 2.0 ** -8
    fast.close()
    ref.close()
