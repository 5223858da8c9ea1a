"""Paged KV cache with per-sequence lengths: ragged batches and continuous
decode, against one oracle run per sequence.

In paged mode every slot of the batch is an independent sequence at its own
position; the oracle runs each sequence alone (batch rows never interact:
dense layers are per row and MoE routing is per token without capacity), so
slot b of a ragged batch must match an oracle batch of that one sequence.
The same configuration with equal lengths must reproduce the contiguous cache
bit for bit (same tiles, same splits, only the addresses differ)."""

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights
from oracle import Oracle
from oracle.sampling import sample as oracle_sample

from parity_util import TOL, GpuRun, assert_parity, compare_moe_steps, compare_steps

pytestmark = pytest.mark.gpu


class Slots:
    """A paged model driven slot by slot, recording every step's outputs."""

    def __init__(self, cfg, w, B, max_len, page_len=64, n_pages=None):
        import torch
        from dual_flow_transformer_decode_b300.model import DualFlowModel
        self.cfg, self.B = cfg, B
        n_pages = n_pages or B * ((max_len + page_len - 1) // page_len)
        self.m = DualFlowModel(cfg, w, max_batch=B, max_len=max_len, page_len=page_len, n_pages=n_pages)
        V, L = cfg.vocab, cfg.n_layers
        dev = "cuda"
        self.lp = torch.zeros(B, V, device=dev)
        self.am = torch.zeros(B, dtype=torch.int32, device=dev)
        self.al = torch.zeros(B, device=dev)
        self.l1 = torch.zeros(B, V, device=dev)
        self.l2 = torch.zeros(B, V, device=dev)
        self.tk = torch.zeros(L, B, max(cfg.aux_k, cfg.top_k, 1), dtype=torch.int32, device=dev)
        self.rl = torch.zeros(L, B, max(cfg.n_experts, 1), device=dev)
        self.m.debug_outputs(self.l1, self.l2, self.tk if cfg.n_experts else None,
                             self.rl if cfg.n_experts else None)
        self.tok = torch.zeros(B, dtype=torch.int32, device=dev)
        self.m.set_batch(B)

    def prefill(self, b, prompt):
        import torch
        self.m.prefill_seq(b, torch.from_numpy(np.ascontiguousarray(prompt, dtype=np.int32)).cuda())

    def step(self, tokens):
        """tokens: host int per slot (free slots: any id)."""
        import torch
        self.tok.copy_(torch.from_numpy(np.asarray(tokens, dtype=np.int32)))
        self.m.decode_step(self.tok, self.lp, self.am, self.al)
        self.m.sync()
        r = {"logp_mix": self.lp.double().cpu().numpy(), "argmax": self.am.cpu().numpy().astype(np.int64),
             "alpha": self.al.double().cpu().numpy(), "logp1": self.l1.double().cpu().numpy()}
        if self.cfg.n_experts:
            r["topk"] = self.tk.cpu().numpy().astype(np.int64)[:, :, :self.cfg.top_k]
            r["router1"] = self.rl.double().cpu().numpy()
        return r

    def close(self):
        self.m.close()


def oracle_sequence(cfg, w, prompt, dec, max_len):
    """One sequence alone: prefill its prompt, decode its tokens."""
    o = Oracle(cfg, w, 1, max_len=max_len)
    o.prefill(np.asarray(prompt)[None, :])
    return o, [o.decode_step(np.array([x])) for x in dec]


def _seq_tokens(cfg, n, seed):
    return dfsynth.tokens(cfg.with_(n_prefill=n, n_steps=0), seed, 1)[0]


def _slot_report(cfg, slot_steps, b, ora_outs):
    """MoE: a routing near tie that the GPU takes the other (valid) way sends
    the token down another computation, so its later values are not compared
    (compare_moe_steps follows each token until such a divergence)."""
    if cfg.n_experts:
        rep = compare_moe_steps(cfg, slot_steps, ora_outs, [b])
        rep["tol"] = TOL[cfg.dtype]
    else:
        rep = compare_steps(cfg, slot_steps, ora_outs, seq_map=[b])
    print("slot", b, {k: v for k, v in rep.items() if not isinstance(v, list) or k == "diverged_at"})
    return rep


def _assert_slots(cfg, reps):
    """Parity over all slots together (the near-tie share is a property of
    the whole comparison, as for a batch)."""
    if cfg.n_experts:
        for k in ("self_inconsistent", "topk_mismatch", "invalid_near_ties", "argmax_mismatch"):
            bad = [x for r in reps for x in r[k]]
            assert not bad, (k, bad[:5])
        assert max(r["max_dlogp_mix"] for r in reps) <= reps[0]["tol"]
        assert max(r["max_dlogp1"] for r in reps) <= reps[0]["tol"]
        compared = sum(r["pairs_compared"] for r in reps)
        assert compared >= 0.5 * (compared + sum(r["pairs_diverged"] for r in reps))
        return
    tot = {"tol": reps[0]["tol"], "decisions": sum(r["decisions"] for r in reps)}
    for k in ("max_dlogp_mix", "max_dlogp1", "max_dalpha", "max_drouter"):
        tot[k] = max(r[k] for r in reps)
    for k in ("argmax_mismatch", "near_ties", "invalid_near_ties", "topk_mismatch"):
        tot[k] = [x for r in reps for x in r[k]]
    assert_parity(cfg, tot)


@pytest.mark.parametrize("name", ["t_bf16", "t_fp32", "t_moe"])
def test_paged_equal_lengths_is_contiguous_bit_for_bit(name, cuda_device):
    cfg = dfsynth.get_config(name).with_(n_steps=3)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    ref = GpuRun(cfg, w, tok)
    import torch
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    B = tok.shape[0]
    m = DualFlowModel(cfg, w, max_batch=B, max_len=cfg.max_len, page_len=64,
                      n_pages=B * ((cfg.max_len + 63) // 64))
    V = cfg.vocab
    lp, l1 = torch.zeros(B, V, device="cuda"), torch.zeros(B, V, device="cuda")
    am = torch.zeros(B, dtype=torch.int32, device="cuda")
    m.debug_outputs(l1)
    tok_d = torch.from_numpy(tok).cuda()
    m.prefill(tok_d[:, :cfg.n_prefill].contiguous())
    for s in range(cfg.n_steps):
        m.decode_step(tok_d[:, cfg.n_prefill + s].contiguous(), lp, am)
        m.sync()
        np.testing.assert_array_equal(lp.double().cpu().numpy(), ref.steps[s]["logp_mix"])
        np.testing.assert_array_equal(l1.double().cpu().numpy(), ref.steps[s]["logp1"])
    n = cfg.n_prefill + cfg.n_steps
    assert m.seq_lengths()[:B] == [n] * B
    for b in range(B):
        np.testing.assert_array_equal(m.seq_kv(b).float().cpu().numpy(), ref.kv[:, :, b, :, :n, :])
    m.close()
    ref.close()


@pytest.mark.parametrize("name,lengths,page_len", [
    ("t_bf16", [150, 37, 64], 64),      # one short, one exactly a page, one spanning 3 pages
    ("t_bf16_b9", [40, 1, 129, 63, 65, 128, 7, 100, 30], 64),
    ("t_fp32", [15, 3], 64),            # the CUDA-core path (fp32)
    ("t_moe", [33, 70, 5, 64, 20], 64),  # token-serial prefill of single slots
    ("t_bf16", [150, 37, 64], 128),
])
def test_ragged_batch_matches_oracle(name, lengths, page_len, cuda_device):
    base = dfsynth.get_config(name)
    S = 4
    max_len = max(lengths) + S + 3
    cfg = base.with_(n_steps=S)
    w = Weights(cfg, 0)
    B = len(lengths)
    seqs = [_seq_tokens(cfg, n + S, 100 + b) for b, n in enumerate(lengths)]
    run = Slots(cfg, w, B, max_len, page_len=page_len)
    for b, n in enumerate(lengths):
        run.prefill(b, seqs[b][:n])
    assert run.m.seq_lengths()[:B] == lengths
    steps = [run.step([seqs[b][lengths[b] + s] for b in range(B)]) for s in range(S)]
    assert run.m.seq_lengths()[:B] == [n + S for n in lengths]
    reps = []
    for b, n in enumerate(lengths):
        o, outs = oracle_sequence(cfg, w, seqs[b][:n], seqs[b][n:n + S], max_len)
        reps.append(_slot_report(cfg, steps, b, outs))
        # the slot's cache against the oracle's, positions 0..n+S-1
        g = run.m.seq_kv(b).double().cpu().numpy()
        for l in range(cfg.n_layers):
            for kind, arr in ((0, o.K), (1, o.V)):
                d = np.abs(g[l, kind] - arr[l][0][:, :n + S])
                assert d.max() < (1e-4 if cfg.dtype == "f32" else 0.05), (b, l, kind, d.max())
    _assert_slots(cfg, reps)
    run.close()


@pytest.mark.parametrize("name,generic", [("t_bf16", False), ("t_bf16", True), ("t_moe", False), ("t_fp32", False)])
def test_continuous_batching(name, generic, cuda_device, monkeypatch):
    """Slots start, finish and restart between steps; every sequence matches
    its own oracle run, so the others are untouched by a release or by a
    prefill into a neighbouring slot (the token-serial prefill of one slot
    computes the other rows too, at their own next positions)."""
    if generic:
        monkeypatch.setenv("DF_FORCE_GENERIC", "1")
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    B, max_len = 3, 140
    # sequence id -> (slot, prompt length, steps, first step at which it runs)
    plan = {0: (0, 40, 2, 0), 1: (1, 70, 7, 0), 2: (2, 10, 4, 1), 3: (0, 90, 5, 2)}
    seqs = {i: _seq_tokens(cfg, n + S, 200 + i) for i, (slot, n, S, _) in plan.items()}
    run = Slots(cfg, w, B, max_len, page_len=64, n_pages=7)
    got = {i: [] for i in plan}
    pos = {}
    total = max(start + S for (_, _, S, start) in plan.values())
    live = {}
    for step in range(total):
        for i, (slot, n, S, start) in plan.items():
            if start == step:
                if slot in live:
                    run.m.release_seq(slot)
                run.prefill(slot, seqs[i][:n])
                live[slot] = i
                pos[i] = n
        toks = [0] * B
        for slot, i in live.items():
            toks[slot] = seqs[i][pos[i]]
        r = run.step(toks)
        for slot, i in list(live.items()):
            got[i].append(r)
            pos[i] += 1
            if len(got[i]) == plan[i][2]:
                run.m.release_seq(slot)
                del live[slot]
    assert run.m.seq_lengths()[:B] == [-1] * B
    reps = []
    for i, (slot, n, S, _) in plan.items():
        assert len(got[i]) == S
        _, outs = oracle_sequence(cfg, w, seqs[i][:n], seqs[i][n:n + S], max_len)
        reps.append(_slot_report(cfg, got[i], slot, outs))
    _assert_slots(cfg, reps)
    run.close()


def test_page_pool_exhaustion_and_reuse(cuda_device):
    from dual_flow_transformer_decode_b300.binding import DFError
    cfg = dfsynth.get_config("t_bf16")
    w = Weights(cfg, 0)
    run = Slots(cfg, w, 2, 200, page_len=64, n_pages=3)
    a, b = _seq_tokens(cfg, 200, 1), _seq_tokens(cfg, 200, 2)
    run.prefill(0, a[:128])              # 2 pages
    with pytest.raises(DFError):
        run.prefill(1, b[:65])           # needs 2, 1 left: refused, slot 1 stays free
    assert run.m.seq_lengths()[:2] == [128, -1]
    run.prefill(1, b[:60])               # 1 page: pool now empty
    # slot 0 at position 128 needs a third page for its next step: refused
    with pytest.raises(DFError):
        run.step([a[128], b[60]])
    assert run.m.seq_lengths()[:2] == [128, 60]
    pages1 = run.m.seq_pages(1)
    run.m.release_seq(1)
    r = run.step([a[128], 0])            # now fits: slot 0 takes the page slot 1 returned
    assert run.m.seq_pages(0)[2] == pages1[0]
    assert run.m.seq_lengths()[:2] == [129, -1]
    _, outs = oracle_sequence(cfg, w, a[:128], a[128:129], 200)
    _assert_slots(cfg, [_slot_report(cfg, [r], 0, outs)])
    run.close()


def test_ragged_generation_draws_at_each_slot_position(cuda_device):
    import torch
    cfg = dfsynth.get_config("t_bf16")
    w = Weights(cfg, 0)
    lengths, S, seed = [150, 37, 64], 4, 77
    max_len = 160
    B = len(lengths)
    seqs = [_seq_tokens(cfg, n + 1, 300 + b) for b, n in enumerate(lengths)]
    run = Slots(cfg, w, B, max_len)
    for b, n in enumerate(lengths):
        run.prefill(b, seqs[b][:n])
    x = torch.tensor([seqs[b][lengths[b]] for b in range(B)], dtype=torch.int32, device="cuda")
    out = torch.zeros(S, B, dtype=torch.int32, device="cuda")
    run.m.generate(x, S, seed, out)
    run.m.sync()
    g = out.cpu().numpy()
    for b, n in enumerate(lengths):
        o = Oracle(cfg, w, 1, max_len=max_len)
        o.prefill(seqs[b][:n][None, :])
        tok = seqs[b][n]
        for s in range(S):
            lp = o.decode_step(np.array([tok]))["logp_mix"][0]
            x_o, margin = oracle_sample(lp, seed, n + s, b)
            if margin > 0.02:
                assert g[s, b] == x_o, (b, s, g[s, b], x_o, margin)
            elif g[s, b] != x_o:
                break
            tok = g[s, b]
    run.close()
