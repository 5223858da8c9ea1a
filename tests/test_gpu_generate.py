"""Generation (sampling from p_mix on the device) against the oracle's
Gumbel-max draws over the same Philox4x64-10 noise.

Each draw is an argmax of log p_mix + g, so it is compared like the argmax:
with eps = max |GPU - oracle| over that row of log p_mix, a draw whose oracle
margin (largest minus second-largest perturbed value) exceeds 2*eps must match
exactly; a smaller margin is a near tie, where the GPU's draw must be a valid
one (its perturbed oracle value within 2*eps of the largest).  A sequence whose
draw legitimately differs at a near tie continues on another token, so it is
compared up to that step only."""

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights
from oracle import Oracle
from oracle.sampling import generate as oracle_generate
from oracle.sampling import gumbel

from parity_util import TOL

pytestmark = pytest.mark.gpu


def _model(cfg, w, tok, aux=True):
    import torch
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    m = DualFlowModel(cfg, w, max_batch=tok.shape[0], max_len=cfg.max_len)
    m.set_mode(aux, False)
    m.prefill(torch.from_numpy(np.ascontiguousarray(tok[:, :cfg.n_prefill])).cuda())
    return m


def _gpu_stepwise(cfg, w, tok, n, seed, aux=True):
    """One df_generate call per step (each fed the previous draw), keeping
    every step's log p_mix."""
    import torch
    m = _model(cfg, w, tok, aux)
    B, V = tok.shape[0], cfg.vocab
    x = torch.from_numpy(np.ascontiguousarray(tok[:, cfg.n_prefill])).cuda()
    out = torch.zeros(1, B, dtype=torch.int32, device="cuda")
    lp = torch.zeros(B, V, device="cuda")
    toks, lps = [], []
    for _ in range(n):
        m.generate(x, 1, seed, out, lp)
        m.sync()
        toks.append(out[0].cpu().numpy().astype(np.int64))
        lps.append(lp.double().cpu().numpy())
        x = out[0].clone()
    m.close()
    return np.stack(toks), lps


def _gpu_oneshot(cfg, w, tok, n, seed, aux=True):
    import torch
    m = _model(cfg, w, tok, aux)
    B = tok.shape[0]
    x = torch.from_numpy(np.ascontiguousarray(tok[:, cfg.n_prefill])).cuda()
    out = torch.zeros(n, B, dtype=torch.int32, device="cuda")
    m.generate(x, n, seed, out)
    m.sync()
    assert m.length == cfg.n_prefill + n
    r = out.cpu().numpy().astype(np.int64)
    m.close()
    return r


@pytest.mark.parametrize("name,aux", [("t_fp32", True), ("t_bf16", True), ("t_bf16_b9", True), ("t_moe", True),
                                      ("t_bf16", False)])
def test_generate_matches_oracle(name, aux, cuda_device):
    cfg = dfsynth.get_config(name)
    n, seed = cfg.n_steps, 20261203
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    g_toks, g_lps = _gpu_stepwise(cfg, w, tok, n, seed, aux)
    # the on-device loop (one call, draws fed back on the device) gives the
    # same draws as the step-by-step calls
    np.testing.assert_array_equal(_gpu_oneshot(cfg, w, tok, n, seed, aux), g_toks)
    o = Oracle(cfg, w, tok.shape[0])
    o.prefill(tok[:, :cfg.n_prefill])
    o_toks, o_margins, o_outs = oracle_generate(o, tok[:, cfg.n_prefill], n, seed, aux=aux)
    tol = TOL[cfg.dtype]
    compared = near = 0
    worst = 0.0
    for b in range(tok.shape[0]):
        for s in range(n):
            ol = o_outs[s]["logp_mix"] if aux else o_outs[s]["logp1"]
            d = np.abs(g_lps[s][b] - ol[b])
            eps = float(d.max())
            worst = max(worst, eps)
            assert eps <= tol, (b, s, eps)
            compared += 1
            if o_margins[s, b] > 2 * eps:
                assert g_toks[s, b] == o_toks[s, b], (b, s, g_toks[s, b], o_toks[s, b], o_margins[s, b], eps)
            else:
                near += 1
                z = ol[b] + gumbel(seed, cfg.n_prefill + s, b, cfg.vocab)
                assert z.max() - z[g_toks[s, b]] <= 2 * eps, (b, s)
                if g_toks[s, b] != o_toks[s, b]:
                    break  # the trajectories part here, both valid
    print(name, "aux" if aux else "primary-only", "draws compared", compared, "near ties", near,
          "max |dlogp_mix|", worst)
    assert near <= max(1, compared // 10)


def test_generate_logp_mix_equals_teacher_forced_step(cuda_device):
    """Drawing does not perturb the distribution: the log p_mix of a generate
    step equals, bit for bit, that of df_decode_step fed the same token."""
    import torch
    cfg = dfsynth.get_config("t_bf16")
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    B, V = tok.shape[0], cfg.vocab
    a = _model(cfg, w, tok)
    b = _model(cfg, w, tok)
    x = torch.from_numpy(np.ascontiguousarray(tok[:, cfg.n_prefill])).cuda()
    out = torch.zeros(2, B, dtype=torch.int32, device="cuda")
    la, lb = torch.zeros(B, V, device="cuda"), torch.zeros(B, V, device="cuda")
    a.generate(x, 1, 7, out, la)
    b.decode_step(x, lb)
    a.sync()
    b.sync()
    assert torch.equal(la, lb)
    a.generate(out[0].clone(), 1, 7, out[1:], la)
    b.decode_step(out[0].clone(), lb)
    a.sync()
    b.sync()
    assert torch.equal(la, lb)
    a.close()
    b.close()


def test_generate_seed_and_capacity(cuda_device):
    import torch
    from dual_flow_transformer_decode_b300.binding import DFError
    cfg = dfsynth.get_config("t_bf16")
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    n = 4
    r1 = _gpu_oneshot(cfg, w, tok, n, 1)
    r2 = _gpu_oneshot(cfg, w, tok, n, 1)
    r3 = _gpu_oneshot(cfg, w, tok, n, 2)
    np.testing.assert_array_equal(r1, r2)
    assert np.mean(r1 != r3) > 0.5
    m = _model(cfg, w, tok)
    B = tok.shape[0]
    x = torch.from_numpy(np.ascontiguousarray(tok[:, cfg.n_prefill])).cuda()
    room = cfg.max_len - cfg.n_prefill
    out = torch.zeros(room + 1, B, dtype=torch.int32, device="cuda")
    with pytest.raises(DFError):
        m.generate(x, room + 1, 3, out)
    assert m.length == cfg.n_prefill
    m.generate(x, 0, 3, out)
    assert m.length == cfg.n_prefill
    m.generate(x, room, 3, out)
    m.sync()
    assert m.length == cfg.max_len
    assert int(out.min()) >= 0 and int(out.max()) < cfg.vocab
    m.close()
