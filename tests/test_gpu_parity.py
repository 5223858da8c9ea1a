"""GPU (C-ABI) vs fp64 oracle parity on small configurations, plus the
GPU-internal bit-exactness toggles (auxiliary flow on/off, grouped/ungrouped)."""

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights

from parity_util import GpuRun, oracle_run, compare_steps, assert_parity, kv_compare, assert_kv_close, tied_weights

pytestmark = pytest.mark.gpu

SMALL = ["t_fp32", "t_fp32_gqa", "t_bf16", "t_bf16_b1", "t_bf16_b9", "t_bf16_long", "t_bf16_b100", "t_bf16_b128",
         "t_bf16_b160", "t_moe", "t_moe_fan"]


@pytest.mark.parametrize("name", SMALL)
def test_parity_small(name, cuda_device):
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok)
    o, outs = oracle_run(cfg, w, tok)
    rep = compare_steps(cfg, g.steps, outs)
    print(name, {k: v for k, v in rep.items() if not isinstance(v, list)})
    assert_parity(cfg, rep)
    mx, rel = kv_compare(cfg, g.kv, o, cfg.max_len, list(range(cfg.batch)))
    print("kv max diff", mx, "relative rms diff", rel)
    assert_kv_close(cfg, mx, rel)
    g.close()


@pytest.mark.parametrize("name", SMALL)
def test_aux_on_off_and_ungrouped_bit_exact(name, cuda_device):
    cfg = dfsynth.get_config(name).with_(n_steps=3)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    on = GpuRun(cfg, w, tok, aux=True)
    off = GpuRun(cfg, w, tok, aux=False)
    ung = GpuRun(cfg, w, tok, aux=True, ungrouped=True)
    np.testing.assert_array_equal(on.kv, off.kv)
    np.testing.assert_array_equal(on.kv, ung.kv)
    for a, b, c in zip(on.steps, off.steps, ung.steps):
        np.testing.assert_array_equal(a["logp1"], b["logp1"])
        np.testing.assert_array_equal(a["logp1"], c["logp1"])
        # aux-off decode reports the primary distribution with alpha = 1
        np.testing.assert_array_equal(b["logp_mix"], b["logp1"])
        assert np.all(b["alpha"] == 1.0)
        # the ungrouped two-pass ablation reaches the same mixture
        np.testing.assert_allclose(a["logp_mix"], c["logp_mix"], rtol=0, atol=1e-5)
        if cfg.n_experts:
            np.testing.assert_array_equal(a["topk"], b["topk"])
            np.testing.assert_array_equal(a["topk"], c["topk"])
    for r in (on, off, ung):
        r.close()


@pytest.mark.parametrize("name", ["t_fp32_gqa", "t_bf16", "t_moe"])
def test_zero_coupling_tied_embeddings_bitwise(name, cuda_device):
    cfg = dfsynth.get_config(name).with_(n_steps=2)
    w = tied_weights(cfg)
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok)
    for r in g.steps:
        np.testing.assert_array_equal(r["logp2"], r["logp1"])
        np.testing.assert_allclose(r["logp_mix"], r["logp1"], rtol=0, atol=2e-6)
    g.close()


def test_host_buffer_step_matches_device_step(cuda_device):
    import torch
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    cfg = dfsynth.get_config("t_bf16").with_(n_steps=2)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    ref = GpuRun(cfg, w, tok)
    m = DualFlowModel(cfg, w)
    m.prefill(torch.from_numpy(tok[:, :cfg.n_prefill].copy()).cuda())
    B, V = cfg.batch, cfg.vocab
    lp = torch.zeros(B, V).pin_memory()
    am = torch.zeros(B, dtype=torch.int32).pin_memory()
    al = torch.zeros(B).pin_memory()
    for s in range(cfg.n_steps):
        t = torch.from_numpy(tok[:, cfg.n_prefill + s].copy()).pin_memory()
        m.decode_step_host(t, lp, am, al)
        np.testing.assert_array_equal(lp.double().numpy(), ref.steps[s]["logp_mix"])
        np.testing.assert_array_equal(am.numpy(), ref.steps[s]["argmax"])
        np.testing.assert_array_equal(al.double().numpy(), ref.steps[s]["alpha"])
    m.close()
    ref.close()


@pytest.mark.parametrize("name,aux,ungrouped", [("t_bf16", True, False), ("t_moe", True, False),
                                               ("t_bf16", False, False), ("t_moe", True, True)])
def test_pipelined_host_steps_match_device_steps(name, aux, ungrouped, cuda_device):
    """df_decode_step_host_async: every step's outputs, copied out on the
    second stream from alternating staging areas, equal the device-buffer
    steps bit for bit (grouped, auxiliary flow off, ungrouped two-pass); a
    synchronous host step in between waits for the pipelined copies of its
    staging area."""
    import torch
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    cfg = dfsynth.get_config(name).with_(n_steps=5)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    ref = GpuRun(cfg, w, tok, aux=aux, ungrouped=ungrouped)
    m = DualFlowModel(cfg, w)
    m.set_mode(aux, ungrouped)
    m.prefill(torch.from_numpy(tok[:, :cfg.n_prefill].copy()).cuda())
    B, V, n = cfg.batch, cfg.vocab, cfg.n_steps
    lp = [torch.full((B, V), float("nan")).pin_memory() for _ in range(n)]
    am = [torch.full((B,), -1, dtype=torch.int32).pin_memory() for _ in range(n)]
    al = [torch.full((B,), float("nan")).pin_memory() for _ in range(n)]
    toks = [torch.from_numpy(tok[:, cfg.n_prefill + s].copy()).pin_memory() for s in range(n)]
    for s in range(3):
        m.decode_step_host_async(toks[s], lp[s], am[s], al[s])
    m.decode_step_host(toks[3], lp[3], am[3], al[3])
    m.decode_step_host_async(toks[4], lp[4], am[4], al[4])
    m.host_wait()
    for s in range(n):
        np.testing.assert_array_equal(lp[s].double().numpy(), ref.steps[s]["logp_mix"])
        np.testing.assert_array_equal(am[s].numpy(), ref.steps[s]["argmax"])
        np.testing.assert_array_equal(al[s].double().numpy(), ref.steps[s]["alpha"])
    m.close()
    ref.close()
