"""GPU vs oracle at the workloads' full sizes, in the launch configuration
bench.py times (max_batch = batch, max_len = prefill + decode steps).

Tolerance: at these depths and widths the bf16 quantisation points turn
the GPU's fp32-level differences into rounding flips that cascade through
the layers; the fp64 oracle itself moves by several 1e-2 in log p when its
pre-rounding values are perturbed by the size of the GPU's own arithmetic
error there (tests/golden/oracle_spread.json, written by
tests/golden/make_oracle_spread.py from the oracle alone).  The
log-probability bound is therefore the larger of the stated bf16 bound
(2e-2) and 1.5 times the largest spread measured that way; the stated 2e-2
holds on the small parity cases (test_gpu_parity.py).

Integer decisions: every argmax whose oracle margin exceeds twice the
measured deviation of its row must match exactly, and such exactly-checked
decisions must make up at least a quarter of all compared ones (so the
check cannot pass vacuously by calling everything a near tie).  Each test
prints one PARITY_RECORD line with what it measured.

The GPU runs the whole batch; the oracle follows sampled sequences (batch
rows are independent: no cross-sequence interaction in dense layers, per-token
routing without capacity in MoE layers).  The 1k-context workload prefills
for real on both sides; longer contexts start from the same seeded synthetic
cache on both sides."""

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights

import json

from parity_util import (GpuRun, oracle_run, oracle_run_synthetic, oracle_follow_synthetic, compare_steps,
                         assert_parity, kv_compare, assert_kv_close, spread_tolerance, kv_spread_bounds)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _weights(cfg):
    w = Weights(cfg, 0)
    w.prefetch()
    return w


def _record(name, rep, tol, spread, **extra):
    """One line with the measured deviations (collected into the design
    notes) and the decision counts; returns it for assertion messages."""
    rec = {"workload": name, "max_dlogp_mix": rep["max_dlogp_mix"], "max_dlogp1": rep["max_dlogp1"],
           "tol": tol, "oracle_spread": spread, "ratio_to_spread": rep["max_dlogp_mix"] / spread if spread else None,
           "argmax_decisions": rep.get("argmax_decisions"), "argmax_exact": rep.get("argmax_exact"),
           "near_ties": len(rep["near_ties"]), **extra}
    line = "PARITY_RECORD " + json.dumps(rec)
    print(line)
    return line


def _assert_exact_floor(rep, line):
    n = rep["argmax_decisions"]
    assert rep["argmax_exact"] >= max(2, n // 4), line


def test_full_tiny_fp32(cuda_device):
    cfg = dfsynth.get_config("tiny_fp32")
    w = _weights(cfg)
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok)
    o, outs = oracle_run(cfg, w, tok)
    rep = compare_steps(cfg, g.steps, outs)
    print({k: v for k, v in rep.items() if not isinstance(v, list)})
    assert_parity(cfg, rep)
    mx, rel = kv_compare(cfg, g.kv, o, cfg.max_len, [0])
    assert_kv_close(cfg, mx, rel)
    g.close()


def test_full_dense1b_ctx1k(cuda_device):
    cfg = dfsynth.get_config("dense1b_ctx1k")
    steps, sample = 6, [0, 5, 10, 15]
    w = _weights(cfg)
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok, steps=steps, keep_kv=False, synth_sample=None)
    kvv = g.m.kv_view()
    gkv = {b: kvv[:, :, b].float().cpu().numpy() for b in sample}
    g.close()
    o, outs = oracle_run(cfg, w, tok[sample], steps=steps)
    rep = compare_steps(cfg, g.steps, outs, seq_map=sample)
    rep["tol"], spread = spread_tolerance(cfg.name, rep["tol"])
    n = cfg.n_prefill + steps
    full = np.zeros((cfg.n_layers, 2, len(sample), cfg.n_kv_heads, n, cfg.head_dim), np.float32)
    for i, b in enumerate(sample):
        full[:, :, i] = gkv[b][:, :, :, :n]
    mx, rel = kv_compare(cfg, full, o, n, list(range(len(sample))))
    kmax, krel = kv_spread_bounds(cfg.name)
    line = _record(cfg.name, rep, rep["tol"], spread, kv_max=mx, kv_rel_rms=rel, kv_bounds=[kmax, krel])
    assert_parity(cfg, rep, max_near_tie_frac=None)
    _assert_exact_floor(rep, line)
    assert mx <= kmax and rel <= krel, line


@pytest.mark.parametrize("name,sample,steps", [
    ("dense1b_ctx32k", [0, 3], 3),
    ("dense24l_b128", [0, 42, 85, 127], 3),
])
def test_full_synthetic_context(name, sample, steps, cuda_device):
    cfg = dfsynth.get_config(name)
    w = _weights(cfg)
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok, steps=steps, keep_kv=False, synth_sample=sample)
    g.close()
    o, outs = oracle_run_synthetic(cfg, w, tok, sample, steps)
    rep = compare_steps(cfg, g.steps, outs, seq_map=sample)
    rep["tol"], spread = spread_tolerance(cfg.name, rep["tol"])
    # the K/V appended by the decode steps
    P = cfg.n_prefill
    mx, ss_d, ss_v = 0.0, 0.0, 0.0
    for i, b in enumerate(sample):
        gnew = g.kv_new[b].astype(np.float64)           # [L][2][Hkv][steps][hd]
        for l in range(cfg.n_layers):
            for kind, arr in ((0, o.K), (1, o.V)):
                d = np.abs(gnew[l, kind] - arr[l][i][:, P:P + steps])
                mx = max(mx, float(d.max()))
                ss_d += float((d * d).sum())
                ss_v += float((arr[l][i][:, P:P + steps] ** 2).sum())
    rel = (ss_d / ss_v) ** 0.5
    kmax, krel = kv_spread_bounds(cfg.name)
    line = _record(cfg.name, rep, rep["tol"], spread, kv_max=mx, kv_rel_rms=rel, kv_bounds=[kmax, krel])
    assert_parity(cfg, rep, max_near_tie_frac=None)
    _assert_exact_floor(rep, line)
    assert mx <= kmax and rel <= krel, line


@pytest.mark.parametrize("name,sample,steps", [
    ("moe64e_top4", [0, 10, 21, 31], 4),
    ("moe64e_top4_aux8", [0, 31], 4),
])
def test_full_moe64e_top4(name, sample, steps, cuda_device):
    """MoE with router replay at full size, and the variant whose auxiliary
    flow adds 4 experts of its own (the same model).  Router-logit
    deviations of the size of the bf16 cascade put some top-k decisions
    inside twice that deviation; at such a near tie the GPU's choice must be
    valid, and the oracle then takes the same one (parity_util.RouteFollower)
    so that every (step, token) pair is compared.  Decisions outside the
    near-tie band must match exactly."""
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    w.prefetch()
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok, steps=steps, keep_kv=False, synth_sample=sample)
    g.close()
    o, outs, route = oracle_follow_synthetic(cfg, w, tok, sample, steps, g.steps)
    rep = compare_steps(cfg, g.steps, outs, seq_map=sample)
    tol, spread = spread_tolerance("moe64e_top4", 2e-2)
    line = _record(name, rep, tol, spread, routing_decisions=route["decisions"], routing_exact=route["exact"],
                   routing_near_ties=len(route["near_ties"]), routing_followed=len(route["followed"]),
                   max_drouter=route["max_drouter"], pairs_compared=len(sample) * steps)
    assert not route["self_inconsistent"], route["self_inconsistent"][:5]
    assert not route["topk_mismatch"], route["topk_mismatch"][:5]
    assert not route["invalid_near_ties"], route["invalid_near_ties"][:5]
    assert not rep["argmax_mismatch"], rep["argmax_mismatch"][:5]
    assert not rep["invalid_near_ties"], rep["invalid_near_ties"][:5]
    assert rep["max_dlogp_mix"] <= tol and rep["max_dlogp1"] <= tol, line
    # most routing decisions lie outside the near-tie band and were checked exactly
    assert route["exact"] >= route["decisions"] // 2, line
    _assert_exact_floor(rep, line)


def test_full_dense1b_ragged_paged_generation(cuda_device):
    """The ragged headline variant in the bench's launch configuration (paged
    cache of 64-position pages, batch 16, prompt lengths from the seeded
    recipe, max_len = longest prompt + 128): every slot prefilled on its own,
    then generation, each step fed the GPU's own draws.  The shortest and
    the longest sequence are followed by the oracle, each alone, with the
    same Philox noise at its own positions; a draw must equal the oracle's
    unless its margin is within twice the measured log p_mix error (then it
    must be a valid draw, and a sequence whose draw differs is followed no
    further).  Tolerance as for dense1b_ctx1k (same model and depth)."""
    import torch
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    from oracle import Oracle
    from oracle.sampling import gumbel, sample as oracle_sample
    cfg = dfsynth.get_config("dense1b_ragged")
    B, PG, steps, seed, span = cfg.batch, cfg.page_len, 3, 11, cfg.n_steps
    lens = dfsynth.prompt_lengths(cfg, 0)
    max_len = int(lens.max()) + span
    n_pages = int(sum((int(n) + span + PG - 1) // PG for n in lens))
    sample = [int(np.argmin(lens)), int(np.argmax(lens))]
    w = _weights(cfg)
    tok = dfsynth.tokens(cfg.with_(n_steps=span), 0)
    m = DualFlowModel(cfg, w, max_batch=B, max_len=max_len, page_len=PG, n_pages=n_pages)
    m.set_batch(B)
    tok_d = torch.from_numpy(tok).cuda()
    for b in range(B):
        m.prefill_seq(b, tok_d[b, :int(lens[b])].contiguous())
    x = torch.tensor([int(tok[b, lens[b]]) for b in range(B)], dtype=torch.int32, device="cuda")
    out = torch.zeros(1, B, dtype=torch.int32, device="cuda")
    lp = torch.zeros(B, cfg.vocab, device="cuda")
    draws, lps = [], []
    for s in range(steps):
        m.generate(x, 1, seed, out, lp)
        m.sync()
        draws.append(out[0].cpu().numpy().astype(np.int64))
        lps.append(lp.double().cpu().numpy())
        x = out[0].clone()
    assert m.seq_lengths()[:B] == [int(n) + steps for n in lens]
    m.close()
    tol, spread = spread_tolerance("dense1b_ctx1k", 2e-2)
    compared = 0
    for b in sample:
        n = int(lens[b])
        o = Oracle(cfg, w, 1, max_len=max_len)
        o.prefill(tok[b:b + 1, :n])
        t_in = int(tok[b, n])
        for s in range(steps):
            lo = o.decode_step(np.array([t_in]))["logp_mix"][0]
            eps = float(np.abs(lps[s][b] - lo).max())
            assert eps <= tol, (b, s, eps, tol)
            x_o, margin = oracle_sample(lo, seed, n + s, b)
            compared += 1
            print("seq", b, "len", n, "step", s, "eps", eps, "margin", margin, "gpu", draws[s][b], "oracle", x_o)
            if margin > 2 * eps:
                assert draws[s][b] == x_o, (b, s)
            else:
                z = lo + gumbel(seed, n + s, b, cfg.vocab)
                assert z.max() - z[draws[s][b]] <= 2 * eps, (b, s)
                if draws[s][b] != x_o:
                    break
            t_in = int(draws[s][b])
    assert compared >= 2
