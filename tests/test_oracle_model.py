"""Model-level pins of the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a structural
property the method fixes (primary flow self-contained, auxiliary flow never
writes the cache), a special case with a closed form, or an independent
standard Transformer assembled from torch library routines.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import dfsynth
from dfsynth.gen import Weights
from oracle import Oracle


def _run(cfg, w, nb=None, steps=None, aux=True, trace=False):
    nb = nb or cfg.batch
    tok = dfsynth.tokens(cfg, 0, nb)
    o = Oracle(cfg, w, nb)
    o.prefill(tok[:, :cfg.n_prefill])
    outs = []
    for s in range(steps or cfg.n_steps):
        outs.append(o.decode_step(tok[:, cfg.n_prefill + s], aux=aux, trace=trace))
    return o, outs


def _tied(cfg, seed=0, a=0.0, b=0.0, c=0.0):
    w = Weights(cfg, seed)
    ov = {("emb2",): w[("emb1",)]}
    for l in range(cfg.n_layers):
        ov[(l, "a")] = np.full(cfg.q_dim, a, np.float32)
        ov[(l, "b")] = np.full(cfg.mlp_hidden, b, np.float32)
        ov[(l, "c")] = np.full(cfg.d_model, c, np.float32)
    return Weights(cfg, seed, overrides=ov)


CFGS = ["t_fp32", "t_fp32_gqa", "t_bf16", "t_moe"]


@pytest.mark.parametrize("name", CFGS)
def test_primary_self_contained_and_aux_writes_no_cache(name):
    cfg = dfsynth.get_config(name).with_(n_steps=3)
    w = Weights(cfg, 0)
    o_on, on = _run(cfg, w, aux=True)
    o_off, off = _run(cfg, w, aux=False)
    for a, b in zip(on, off):
        np.testing.assert_array_equal(a["logp1"], b["logp1"])
        np.testing.assert_array_equal(a["topk"], b["topk"])
    for l in range(cfg.n_layers):
        for s in range(cfg.batch):
            np.testing.assert_array_equal(o_on.K[l][s], o_off.K[l][s])
            np.testing.assert_array_equal(o_on.V[l][s], o_off.V[l][s])
    # nothing beyond position t was touched
    assert np.all(o_on.K[0][0][:, o_on.t:] == 0)


@pytest.mark.parametrize("name", CFGS)
def test_zero_coupling_tied_embeddings_collapses_to_primary(name):
    cfg = dfsynth.get_config(name).with_(n_steps=2)
    _, outs = _run(cfg, _tied(cfg))
    for r in outs:
        np.testing.assert_array_equal(r["logp2"], r["logp1"])
        np.testing.assert_allclose(r["logp_mix"], r["logp1"], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(r["argmax"], r["argmax1"])


@pytest.mark.parametrize("name", CFGS)
def test_alpha_at_least_half(name):
    cfg = dfsynth.get_config(name).with_(n_steps=2)
    _, outs = _run(cfg, Weights(cfg, 0))
    for r in outs:
        assert np.all(r["alpha"] >= 0.5) and np.all(r["alpha"] <= 1.0)
        np.testing.assert_allclose(np.exp(r["logp_mix"]).sum(1), 1.0, atol=1e-12)
        p1 = np.exp(r["logp1"])
        np.testing.assert_allclose(r["alpha"], 0.5 + 0.5 * (p1 * p1).sum(1), rtol=1e-14)


def test_alpha_spans_range_with_peaked_head():
    cfg = dfsynth.get_config("t_fp32").with_(n_steps=4, lm_scale=60.0)
    _, outs = _run(cfg, Weights(cfg, 0))
    al = np.concatenate([r["alpha"] for r in outs])
    assert al.min() >= 0.5 and al.max() > 0.6


def test_query_coupling_minus_one_gives_uniform_attention():
    # E2 = E1 and a = -1: in layer 0 the auxiliary pre-RoPE query equals
    # q1 - q1 = 0, so its attention is the plain average of V[0..t].
    cfg = dfsynth.get_config("t_fp32_gqa").with_(n_steps=2)
    o, outs = _run(cfg, _tied(cfg, a=-1.0), trace=True)
    t = outs[-1]["t"]
    tr = outs[-1]["trace"][0]
    assert np.all(tr["Q2"] == 0)
    G = cfg.group
    for s in range(cfg.batch):
        for h in range(cfg.n_heads):
            mean_v = o.V[0][s][h // G, :t + 1].mean(axis=0)
            np.testing.assert_allclose(tr["o2"][s].reshape(cfg.n_heads, -1)[h], mean_v, atol=1e-13)


@pytest.mark.parametrize("name", ["t_fp32_gqa", "t_moe"])
@pytest.mark.parametrize("which", ["b", "c"])
def test_mlp_couplings_minus_one_cancel_layer0_mlp(name, which):
    # E2 = E1, a = 0: in layer 0 both flows carry the same state.  b = -1
    # cancels the auxiliary MLP intermediate (z2 = z1 - z1); c = -1 cancels its
    # MLP output (y2 = y1 - y1).  Either way the layer-0 MLP adds nothing to h2.
    cfg = dfsynth.get_config(name).with_(n_steps=1)
    kw = {which: -1.0}
    _, outs = _run(cfg, _tied(cfg, **kw), trace=True)
    tr = outs[0]["trace"][0]
    np.testing.assert_allclose(tr["h2"], tr["h2_attn"], rtol=0, atol=1e-12)
    # and a layer-0 MLP that is not cancelled does change h2
    _, outs0 = _run(cfg, _tied(cfg), trace=True)
    assert np.abs(outs0[0]["trace"][0]["h2"] - outs0[0]["trace"][0]["h2_attn"]).max() > 1e-4


def test_moe_single_expert_reduces_to_dense():
    moe = dfsynth.get_config("t_moe").with_(n_experts=1, top_k=1, n_steps=2)
    dense = moe.with_(n_experts=0, top_k=0, ffn_hidden=moe.expert_hidden, expert_hidden=0)
    wm = Weights(moe, 0)
    ov = {}
    for l in range(moe.n_layers):
        for n in ("wg", "wu", "wd"):
            ov[(l, n)] = wm[(l, 0, n)]
        ov[(l, "b")] = wm[(l, "b")]
    wd = Weights(dense, 0, overrides=ov)
    _, om = _run(moe, wm)
    _, od = _run(dense, wd)
    for a, b in zip(om, od):
        np.testing.assert_allclose(a["logp_mix"], b["logp_mix"], rtol=0, atol=1e-12)
        assert np.all(a["topk"] == 0)


def test_moe_replay_gates_are_normalised_and_shared_set():
    cfg = dfsynth.get_config("t_moe").with_(n_steps=2)
    o, outs = _run(cfg, Weights(cfg, 0))
    for r in outs:
        k = r["topk"]
        assert k.shape == (cfg.n_layers, cfg.batch, cfg.top_k)
        for l in range(cfg.n_layers):
            for s in range(cfg.batch):
                assert len(set(k[l, s])) == cfg.top_k
                # descending router logits
                rl = r["router1"][l][s][k[l, s]]
                assert np.all(np.diff(rl) <= 0)


@pytest.mark.parametrize("name", CFGS)
def test_token_serial_decode_equals_prefill(name):
    # Two code paths of the oracle: the causal-mask prefill over n positions,
    # and n primary-only steps one position at a time, must write the same KV.
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    n = 12
    a = Oracle(cfg, w, cfg.batch)
    a.prefill(tok[:, :n])
    b = Oracle(cfg, w, cfg.batch)
    b.prefill(tok[:, :1])
    for p in range(1, n):
        b.decode_step(tok[:, p], aux=False)
    for l in range(cfg.n_layers):
        for s in range(cfg.batch):
            np.testing.assert_allclose(a.K[l][s][:, :n], b.K[l][s][:, :n], rtol=0, atol=1e-12)
            np.testing.assert_allclose(a.V[l][s][:, :n], b.V[l][s][:, :n], rtol=0, atol=1e-12)


def _torch_standard_transformer(cfg, w, tok):
    """A standard pre-norm causal Transformer over tok[n] from torch library
    routines (rms_norm, scaled_dot_product_attention, silu, log_softmax); RoPE
    as a complex rotation of (i, i + hd/2) pairs.  Returns (last-position
    log-probs, K[l][Hkv][n][hd], V[l])."""
    T = lambda k: torch.from_numpy(np.asarray(w[k], dtype=np.float64))
    n = len(tok)
    hd, Hq, Hkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    x = T(("emb1",))[torch.from_numpy(tok.astype(np.int64))]
    pos = torch.arange(n, dtype=torch.float64)
    inv = cfg.rope_theta ** (-torch.arange(hd // 2, dtype=torch.float64) * 2 / hd)
    rot = torch.polar(torch.ones(n, hd // 2, dtype=torch.float64), pos[:, None] * inv[None])

    def rope_c(v):  # v [H][n][hd]
        z = torch.complex(v[..., : hd // 2], v[..., hd // 2:]) * rot
        return torch.cat([z.real, z.imag], -1)

    Ks, Vs = [], []
    for l in range(cfg.n_layers):
        u = F.rms_norm(x, (cfg.d_model,), weight=T((l, "attn_norm")), eps=cfg.norm_eps)
        q = (u @ T((l, "wq")).T).view(n, Hq, hd).transpose(0, 1)
        k = (u @ T((l, "wk")).T).view(n, Hkv, hd).transpose(0, 1)
        v = (u @ T((l, "wv")).T).view(n, Hkv, hd).transpose(0, 1)
        q, k = rope_c(q), rope_c(k)
        Ks.append(k.numpy())
        Vs.append(v.numpy())
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, enable_gqa=True)[0]
        x = x + o.transpose(0, 1).reshape(n, -1) @ T((l, "wo")).T
        u = F.rms_norm(x, (cfg.d_model,), weight=T((l, "mlp_norm")), eps=cfg.norm_eps)
        x = x + (F.silu(u @ T((l, "wg")).T) * (u @ T((l, "wu")).T)) @ T((l, "wd")).T
    u = F.rms_norm(x, (cfg.d_model,), weight=T(("final_norm",)), eps=cfg.norm_eps)
    return torch.log_softmax(u[-1] @ T(("lm_head",)).T, -1).numpy(), Ks, Vs


@pytest.mark.parametrize("name", ["t_fp32", "t_fp32_gqa"])
def test_primary_flow_is_a_standard_transformer(name):
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    P = cfg.n_prefill + 1
    o = Oracle(cfg, w, cfg.batch)
    o.prefill(tok[:, :P - 1])
    r = o.decode_step(tok[:, P - 1], aux=True)
    for s in range(cfg.batch):
        lp, Ks, Vs = _torch_standard_transformer(cfg, w, tok[s, :P])
        np.testing.assert_allclose(r["logp1"][s], lp, rtol=0, atol=1e-11)
        for l in range(cfg.n_layers):
            np.testing.assert_allclose(o.K[l][s][:, :P], Ks[l], rtol=0, atol=1e-12)
            np.testing.assert_allclose(o.V[l][s][:, :P], Vs[l], rtol=0, atol=1e-12)


def _bf16_by_hand(x):
    """Round fp64 values to the nearest bf16 value, ties to even, in one
    rounding: frexp gives x = m * 2^e with 0.5 <= |m| < 1, so m * 256 carries
    exactly bf16's 8 significant bits before the point; torch.round rounds
    half to even."""
    m, e = torch.frexp(x)
    return torch.ldexp(torch.round(m * 256.0) / 256.0, e)


def _torch_dualflow_bf16(cfg, w, tok):
    """Both flows at the last position of tok[n], written out with torch
    library routines, with every bf16 rounding inserted by hand where the
    method's bf16 storage puts it: GEMM inputs (normed rows, attention
    output, MLP hidden), cache stores (K after RoPE, V) and the queries
    entering attention (after RoPE); residual, norms, couplings, softmax and
    mixture stay in fp64.  The primary flow runs causally over all n
    positions; the auxiliary flow runs at the last one only, from E2, with
    Q2 = Wq u2 + a * q1 (q1 the primary's unrounded pre-RoPE query there),
    z2 += b * z1 (post-gating, unrounded z1), y2 += c * y1 (before the
    residual add), attending to the primary's K/V 0..n-1.
    Returns (log p1, log p2, log p_mix, alpha, K[l], V[l])."""
    T = lambda k: torch.from_numpy(np.asarray(w[k], dtype=np.float64))  # noqa: E731
    bf = _bf16_by_hand
    n = len(tok)
    hd, Hq, Hkv, d = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.d_model
    x1 = T(("emb1",))[torch.from_numpy(tok.astype(np.int64))]
    x2 = T(("emb2",))[int(tok[-1])].clone()
    pos = torch.arange(n, dtype=torch.float64)
    inv = cfg.rope_theta ** (-torch.arange(hd // 2, dtype=torch.float64) * 2 / hd)
    rot = torch.polar(torch.ones(n, hd // 2, dtype=torch.float64), pos[:, None] * inv[None])

    def rope_c(v, r):  # v [..][hd] rotated by r [..][hd/2]
        z = torch.complex(v[..., : hd // 2], v[..., hd // 2:]) * r
        return torch.cat([z.real, z.imag], -1)

    def norm(x, key):
        return F.rms_norm(x, (d,), weight=T(key), eps=cfg.norm_eps)

    Ks, Vs = [], []
    for l in range(cfg.n_layers):
        u = bf(norm(x1, (l, "attn_norm")))
        q = u @ T((l, "wq")).T                                            # [n][Hq*hd], pre-RoPE
        k = (u @ T((l, "wk")).T).view(n, Hkv, hd).transpose(0, 1)
        v = (u @ T((l, "wv")).T).view(n, Hkv, hd).transpose(0, 1)
        kr, vr = bf(rope_c(k, rot)), bf(v)
        Ks.append(kr.numpy())
        Vs.append(vr.numpy())
        qr = bf(rope_c(q.view(n, Hq, hd).transpose(0, 1), rot))
        o1 = F.scaled_dot_product_attention(qr[None], kr[None], vr[None], is_causal=True, enable_gqa=True)[0]
        u2 = bf(norm(x2, (l, "attn_norm")))
        Q2 = u2 @ T((l, "wq")).T + T((l, "a")) * q[-1]
        q2r = bf(rope_c(Q2.view(Hq, 1, hd), rot[-1:]))
        o2 = F.scaled_dot_product_attention(q2r[None], kr[None], vr[None], enable_gqa=True)[0]
        x1 = x1 + bf(o1.transpose(0, 1).reshape(n, -1)) @ T((l, "wo")).T
        x2 = x2 + bf(o2.reshape(-1)) @ T((l, "wo")).T
        u = bf(norm(x1, (l, "mlp_norm")))
        z1 = F.silu(u @ T((l, "wg")).T) * (u @ T((l, "wu")).T)
        y1 = bf(z1) @ T((l, "wd")).T
        x1 = x1 + y1
        u2 = bf(norm(x2, (l, "mlp_norm")))
        z2 = F.silu(u2 @ T((l, "wg")).T) * (u2 @ T((l, "wu")).T) + T((l, "b")) * z1[-1]
        x2 = x2 + bf(z2) @ T((l, "wd")).T + T((l, "c")) * y1[-1]
    lp1 = torch.log_softmax(bf(norm(x1[-1], ("final_norm",))) @ T(("lm_head",)).T, -1)
    lp2 = torch.log_softmax(bf(norm(x2, ("final_norm",))) @ T(("lm_head",)).T, -1)
    alpha = 0.5 + 0.5 * torch.exp(2 * lp1).sum()
    lmix = torch.logaddexp(torch.log(alpha) + lp1, torch.log1p(-alpha) + lp2)
    return lp1.numpy(), lp2.numpy(), lmix.numpy(), float(alpha), Ks, Vs


def test_bf16_by_hand_rounds_once_to_nearest_even():
    # the test's own rounding, against values whose bf16 neighbours are known
    one = 1.0
    ulp = 2.0 ** -7                                   # bf16 spacing in [1, 2)
    x = torch.tensor([one + ulp / 2, one + 1.5 * ulp, one + ulp / 2 + 2.0 ** -40, -(one + ulp / 2),
                      3.0 * 2.0 ** -130, 0.0], dtype=torch.float64)
    want = [one, one + 2 * ulp, one + ulp, -one, 3.0 * 2.0 ** -130, 0.0]
    assert _bf16_by_hand(x).tolist() == want
    r = torch.randn(10000, dtype=torch.float64) * 7
    # single rounding agrees with fp32 -> bf16 wherever fp64 -> fp32 is exact
    r32 = r.float().double()
    assert torch.equal(_bf16_by_hand(r32), r32.float().to(torch.bfloat16).double())


@pytest.mark.parametrize("name", ["t_bf16", "t_bf16_b9"])
def test_bf16_rounding_points_match_a_hand_written_dual_flow_step(name):
    """The oracle in bf16 mode against the step written out above with the
    bf16 roundings placed by hand: a rounding point missing, added or moved
    (for instance the query rounded before RoPE, or the coupling reading a
    rounded q1 or z1) changes log p by far more than the tolerance, which
    only has to absorb fp64 summation order."""
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    P = cfg.n_prefill + 1
    o = Oracle(cfg, w, cfg.batch)
    o.prefill(tok[:, :P - 1])
    r = o.decode_step(tok[:, P - 1], aux=True)
    for s in range(cfg.batch):
        lp1, lp2, lmix, alpha, Ks, Vs = _torch_dualflow_bf16(cfg, w, tok[s, :P])
        np.testing.assert_allclose(r["logp1"][s], lp1, rtol=0, atol=1e-9)
        np.testing.assert_allclose(r["logp2"][s], lp2, rtol=0, atol=1e-9)
        np.testing.assert_allclose(r["logp_mix"][s], lmix, rtol=0, atol=1e-9)
        assert abs(r["alpha"][s] - alpha) <= 1e-12
        for l in range(cfg.n_layers):
            np.testing.assert_array_equal(o.K[l][s][:, :P], Ks[l])
            np.testing.assert_array_equal(o.V[l][s][:, :P], Vs[l])


# ---------------------------------------------------------------- auxiliary fan-out

def _aux_moe_layer0_by_hand(cfg, w, tr_primary, tr_aux, nx_pick):
    """Layer 0's auxiliary MoE written out independently of the oracle's
    routing code: the primary set by sorting, the auxiliary extras by
    `nx_pick(r2, S)`, softmax over the union, b coupling only on the
    replayed experts, c coupling of the primary output.  Returns h2 after
    the layer."""
    bf = lambda x: x  # noqa: E731 — fp32 parity config: no rounding points
    if cfg.dtype == "bf16":
        from oracle import bf16_rne as bf
    d = cfg.d_model

    def rms(x, g):
        return x / np.sqrt(np.mean(x * x) + cfg.norm_eps) * g

    def hidden(e, u):
        wg = np.asarray(w[(0, e, "wg")], np.float64)
        wu = np.asarray(w[(0, e, "wu")], np.float64)
        a, b = wg @ u, wu @ u
        return a / (1 + np.exp(-a)) * b

    g_mlp = np.asarray(w[(0, "mlp_norm")], np.float64)
    Wr = np.asarray(w[(0, "router")], np.float64)
    bvec = np.asarray(w[(0, "b")], np.float64)
    cvec = np.asarray(w[(0, "c")], np.float64)
    out = []
    for s in range(tr_aux[0]["h2_attn"].shape[0]):
        h1 = tr_primary[0]["h1_attn"][s]
        h2 = tr_aux[0]["h2_attn"][s]
        r1 = Wr @ rms(h1, g_mlp)
        S = sorted(range(cfg.n_experts), key=lambda e: (-r1[e], e))[:cfg.top_k]
        u1 = bf(rms(h1, g_mlp))
        p1 = np.exp(r1[S] - r1[S].max())
        p1 /= p1.sum()
        z1 = {e: hidden(e, u1) for e in S}
        y1 = sum(p1[j] * (np.asarray(w[(0, e, "wd")], np.float64) @ bf(z1[e])) for j, e in enumerate(S))
        r2 = Wr @ rms(h2, g_mlp)
        SA = list(S) + list(nx_pick(r2, S))
        p2 = np.exp(r2[SA] - r2[SA].max())
        p2 /= p2.sum()
        u2 = bf(rms(h2, g_mlp))
        y2 = np.zeros(d)
        for j, e in enumerate(SA):
            z = hidden(e, u2) + (bvec * z1[e] if e in S else 0.0)
            y2 += p2[j] * (np.asarray(w[(0, e, "wd")], np.float64) @ bf(z))
        out.append(h2 + y2 + cvec * y1)
    return np.stack(out)


@pytest.mark.parametrize("aux_top_k", [4, 8])
def test_aux_fanout_layer_written_out(aux_top_k):
    """Independent fan-out: the oracle's auxiliary MoE layer against the same
    layer written out by hand — the extras are the largest auxiliary router
    logits outside the replayed set (aux_top_k = E: every expert, a dense
    softmax mixture), gates are a softmax over the union, and only replayed
    experts carry the b coupling."""
    cfg = dfsynth.get_config("t_moe").with_(n_layers=1, n_steps=1, aux_top_k=aux_top_k, dtype="f32")
    w = Weights(cfg, 0)
    _, outs = _run(cfg, w, trace=True)
    r = outs[0]
    nx = aux_top_k - cfg.top_k

    def pick(r2, S):
        rest = [e for e in range(cfg.n_experts) if e not in S]
        return sorted(rest, key=lambda e: (-r2[e], e))[:nx]

    ref = _aux_moe_layer0_by_hand(cfg, w, r["trace_primary"], r["trace"], pick)
    np.testing.assert_allclose(r["trace"][0]["h2"], ref, rtol=1e-10, atol=1e-12)
    assert r["topk_aux"].shape == (1, cfg.batch, nx)
    for s in range(cfg.batch):
        assert not set(r["topk_aux"][0, s]) & set(r["topk"][0, s])


def test_aux_fanout_equal_to_top_k_is_replay():
    """aux_top_k = top_k: exactly the router-replay model."""
    cfg = dfsynth.get_config("t_moe").with_(n_steps=2)
    w = Weights(cfg, 0)
    _, a = _run(cfg, w)
    _, b = _run(cfg.with_(aux_top_k=cfg.top_k), w)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x["logp_mix"], y["logp_mix"])


def test_aux_fanout_leaves_primary_unchanged():
    """The auxiliary flow's extra experts change nothing the primary computes
    (cache, primary log-probabilities, primary sets)."""
    cfg = dfsynth.get_config("t_moe_fan").with_(n_steps=2)
    w = Weights(cfg, 0)
    oa, a = _run(cfg, w)
    ob, b = _run(cfg.with_(aux_top_k=0), w)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x["logp1"], y["logp1"])
        np.testing.assert_array_equal(x["topk"], y["topk"])
        assert not np.array_equal(x["logp2"], y["logp2"])
    for l in range(cfg.n_layers):
        for s in range(cfg.batch):
            np.testing.assert_array_equal(oa.K[l][s], ob.K[l][s])
