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


@pytest.mark.parametrize("name", ["t_bf16", "t_bf16_b9", "t_moe", "t_moe_fan"])
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
        if "topk_aux" in a:
            # the auxiliary flow's own experts: same decisions unless near a tie
            print("  own-expert sets equal:", float(np.mean(np.sort(a["topk_aux"], -1) == np.sort(b["topk_aux"], -1))))
    diff = np.abs(fast.kv - ref.kv).astype(np.float64)
    rel = float(np.sqrt((diff ** 2).sum() / (ref.kv.astype(np.float64) ** 2).sum()))
    print("kv max", diff.max(), "relative rms", rel)
    assert diff.max() < 0.05 and rel < 2.0 ** -8
    fast.close()
    ref.close()


@pytest.mark.parametrize("name,aux,ungrouped", [("t_bf16", True, False), ("t_bf16_b9", True, False),
                                                ("t_bf16_long", True, False), ("t_bf16", False, False),
                                                ("t_bf16", True, True)])
def test_persistent_kernel_matches_kernel_sequence(name, aux, ungrouped, cuda_device):
    """The one-launch persistent pass (opt-in with DF_MK=1; dense bf16, up to
    32 stacked rows) against the per-layer kernel sequence of the same
    library: prefill and decode, both flows, aux-off and the two-pass
    ungrouped mode."""
    cfg = dfsynth.get_config(name).with_(n_steps=3)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    ref = GpuRun(cfg, w, tok, aux=aux, ungrouped=ungrouped)
    os.environ["DF_MK"] = "1"
    try:
        mk = GpuRun(cfg, w, tok, aux=aux, ungrouped=ungrouped)
    finally:
        del os.environ["DF_MK"]
    # one launch for all layers of a pass instead of seven per layer
    print("kernels per step", mk.m.step_kernels, ref.m.step_kernels)
    assert 0 < mk.m.step_kernels < ref.m.step_kernels
    for a, b in zip(mk.steps, ref.steps):
        d1 = np.abs(a["logp1"] - b["logp1"]).max()
        dm = np.abs(a["logp_mix"] - b["logp_mix"]).max()
        print(name, aux, ungrouped, "max |dlogp1|", d1, "max |dlogp_mix|", dm)
        assert d1 < 5e-3 and dm < 5e-3
        if aux:
            d2 = np.abs(a["logp2"] - b["logp2"]).max()
            assert d2 < 5e-3, d2
    diff = np.abs(mk.kv - ref.kv).astype(np.float64)
    rel = float(np.sqrt((diff ** 2).sum() / (ref.kv.astype(np.float64) ** 2).sum()))
    print("kv max", diff.max(), "relative rms", rel)
    assert diff.max() < 0.05 and rel < 2.0 ** -8
    mk.close()
    ref.close()
