"""Pins of the fp64 oracle's building blocks to closed forms, special cases and
library routines (CPU only)."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import bf16_rne, rmsnorm, silu, rope, attend, log_softmax, mixture, topk_desc


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_ties_to_even():
    # quantum near 1 is 2^-7: 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert bf16_rne(1.0 + 2 ** -8) == 1.0
    assert bf16_rne(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6
    assert bf16_rne(-(1.0 + 3 * 2 ** -8)) == -(1.0 + 2 ** -6)
    # a value just above a tie must round up; rounding through fp32 first
    # would land exactly on the tie and round down
    assert bf16_rne(1.0 + 2 ** -8 + 2 ** -40) == 1.0 + 2 ** -7
    assert bf16_rne(0.0) == 0.0


def test_bf16_matches_torch_on_fp32_inputs():
    g = np.random.default_rng(1)
    x = np.concatenate([g.standard_normal(20000) * s for s in (1e-30, 1e-3, 1.0, 1e3, 1e30)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(bf16_rne(x.astype(np.float64)), ref)


def test_bf16_subnormal_quantum():
    q = 2.0 ** -133
    assert bf16_rne(3 * q) == 3 * q
    assert bf16_rne(2.5 * q) == 2 * q      # tie -> even
    assert bf16_rne(3.5 * q) == 4 * q


# ---------------------------------------------------------------- rmsnorm / silu

def test_rmsnorm_closed_form():
    out = rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(out, [3 / r, 8 / r], rtol=0, atol=1e-15)
    out = rmsnorm(np.array([0.0, 0.0, 0.0]), np.ones(3), 1e-5)
    assert np.all(out == 0)


def test_rmsnorm_matches_torch():
    g = np.random.default_rng(2)
    x = g.standard_normal((7, 96))
    w = 1 + 0.1 * g.standard_normal(96)
    ref = F.rms_norm(torch.from_numpy(x), (96,), weight=torch.from_numpy(w), eps=1e-5).numpy()
    np.testing.assert_allclose(rmsnorm(x, w, 1e-5), ref, rtol=1e-13, atol=1e-14)


def test_silu():
    assert silu(0.0) == 0.0
    np.testing.assert_allclose(silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    x = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-14, atol=1e-300)


# ---------------------------------------------------------------- rope

def test_rope_identity_at_zero():
    x = np.random.default_rng(3).standard_normal((5, 64))
    np.testing.assert_array_equal(rope(x, 0, 1e4), x)


def test_rope_two_dims_is_rotation_by_t():
    x = np.array([0.3, -1.7])
    for t in (1, 5, 123):
        c, s = math.cos(t), math.sin(t)
        np.testing.assert_allclose(rope(x, t, 1e4), [0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s], atol=1e-14)


def test_rope_is_complex_rotation_of_half_pairs():
    g = np.random.default_rng(4)
    hd, theta, t = 32, 1e4, 77
    x = g.standard_normal(hd)
    z = x[: hd // 2] + 1j * x[hd // 2:]
    ang = t * theta ** (-np.arange(hd // 2) * 2.0 / hd)
    zr = z * np.exp(1j * ang)
    np.testing.assert_allclose(rope(x, t, theta), np.concatenate([zr.real, zr.imag]), atol=1e-13)


def test_rope_preserves_pair_norms_and_scores_depend_on_offset():
    g = np.random.default_rng(5)
    q, k = g.standard_normal(64), g.standard_normal(64)
    a = rope(q, 10, 1e4) @ rope(k, 3, 1e4)
    b = rope(q, 1010, 1e4) @ rope(k, 1003, 1e4)
    np.testing.assert_allclose(a, b, rtol=1e-10)
    r = rope(q, 999, 1e4)
    np.testing.assert_allclose(r[:32] ** 2 + r[32:] ** 2, q[:32] ** 2 + q[32:] ** 2, rtol=1e-12)


# ---------------------------------------------------------------- attention

def _brute_attention(q, K, V):
    Hq, hd = len(q), len(q[0])
    Hkv = len(K)
    G = Hq // Hkv
    out = []
    for h in range(Hq):
        kh = K[h // G]
        scores = [sum(q[h][i] * kh[j][i] for i in range(hd)) / math.sqrt(hd) for j in range(len(kh))]
        m = max(scores)
        w = [math.exp(s - m) for s in scores]
        tot = sum(w)
        out.append([sum(w[j] / tot * V[h // G][j][i] for j in range(len(kh))) for i in range(hd)])
    return out


@pytest.mark.parametrize("Hq,Hkv,n", [(2, 2, 1), (4, 2, 5), (6, 3, 8), (4, 1, 7)])
def test_attention_vs_brute_force(Hq, Hkv, n):
    g = np.random.default_rng(10 + n)
    hd = 4
    q = g.standard_normal((Hq, hd))
    K = g.standard_normal((Hkv, n, hd))
    V = g.standard_normal((Hkv, n, hd))
    ref = np.array(_brute_attention(q.tolist(), K.tolist(), V.tolist()))
    np.testing.assert_allclose(attend(q, K, V), ref, rtol=0, atol=1e-12)


def test_attention_single_position_returns_value():
    g = np.random.default_rng(6)
    q = g.standard_normal((4, 8)) * 10
    K = g.standard_normal((2, 1, 8))
    V = g.standard_normal((2, 1, 8))
    o = attend(q, K, V)
    for h in range(4):
        np.testing.assert_array_equal(o[h], V[h // 2, 0])


def test_attention_matches_torch_sdpa_gqa():
    g = np.random.default_rng(7)
    Hq, Hkv, n, hd = 8, 2, 33, 16
    q = g.standard_normal((Hq, hd))
    K = g.standard_normal((Hkv, n, hd))
    V = g.standard_normal((Hkv, n, hd))
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        enable_gqa=True)[0, :, 0].numpy()
    np.testing.assert_allclose(attend(q, K, V), ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- softmax / mixture / top-k

def test_log_softmax():
    z = np.array([0.0, math.log(3.0)])
    np.testing.assert_allclose(log_softmax(z), [math.log(0.25), math.log(0.75)], atol=1e-15)
    x = np.random.default_rng(8).standard_normal((3, 1000)) * 5
    np.testing.assert_allclose(log_softmax(x), torch.log_softmax(torch.from_numpy(x), -1).numpy(), atol=1e-13)


def test_mixture_closed_form_two_symbols():
    # p1 = (1/2, 1/2): sum p1^2 = 1/2 -> alpha = 3/4; p2 = (1, 0)
    lp1 = np.log([0.5, 0.5])
    lp2 = np.array([0.0, -np.inf])
    lm, a = mixture(lp1, lp2)
    assert a == 0.75
    np.testing.assert_allclose(np.exp(lm), [0.625, 0.375], atol=1e-15)


def test_mixture_alpha_bounds():
    V = 1000
    lm, a = mixture(np.full(V, -math.log(V)), np.full(V, -math.log(V)))
    np.testing.assert_allclose(a, 0.5 + 0.5 / V, rtol=1e-14)
    one_hot = np.full(V, -np.inf)
    one_hot[17] = 0.0
    lm, a = mixture(one_hot, np.log(np.full(V, 1.0 / V)))
    assert a == 1.0 and np.argmax(lm) == 17 and lm[17] == 0.0
    g = np.random.default_rng(9)
    for scale in (0.1, 1, 5, 30):
        lp1 = log_softmax(g.standard_normal(V) * scale)
        lp2 = log_softmax(g.standard_normal(V) * scale)
        lm, a = mixture(lp1, lp2)
        assert 0.5 <= a <= 1.0
        assert abs(np.exp(lm).sum() - 1.0) < 1e-12


def test_topk_desc_ties_go_to_lower_index():
    r = np.array([0.5, 2.0, 0.5, 2.0, 1.0, 0.5])
    np.testing.assert_array_equal(topk_desc(r, 4), [1, 3, 4, 0])
    g = np.random.default_rng(11)
    for _ in range(50):
        r = np.round(g.standard_normal(64), 1)
        np.testing.assert_array_equal(topk_desc(r, 4), np.argsort(-r, kind="stable")[:4])


def test_aux_own_experts_are_the_next_ranks_after_the_replayed_set():
    """The auxiliary flow's own experts (independent fan-out): with S the
    primary top-k of the same logits they are ranks k .. k+nx-1 of one stable
    descending sort; for any other S, brute force over all subsets of the
    right size that avoid S picks the same set (largest logit sum, then the
    lexicographically smallest index list).  The reported margin is the gap
    at the cut."""
    from itertools import combinations
    from oracle import Oracle
    g = np.random.default_rng(12)
    for _ in range(40):
        r = np.round(g.standard_normal(12), 1)  # coarse values: many ties
        order = np.argsort(-r, kind="stable")
        for k, nx in ((2, 2), (4, 4), (1, 6)):
            S = topk_desc(r, k)
            X = Oracle._aux_extra(r, S, nx)
            np.testing.assert_array_equal(X, order[k:k + nx])
            assert Oracle._aux_extra_margin(r, S, nx) == r[order[k + nx - 1]] - r[order[k + nx]]
        S = g.choice(12, size=3, replace=False)
        rest = [e for e in range(12) if e not in set(S.tolist())]
        best = min(combinations(rest, 3), key=lambda c: (-sum(r[e] for e in c), sorted(c)))
        X = Oracle._aux_extra(r, S, 3)
        assert sorted(X.tolist()) == sorted(best)
        assert not set(X.tolist()) & set(S.tolist())
        assert all(r[X[i]] >= r[X[i + 1]] for i in range(len(X) - 1))
    assert Oracle._aux_extra(r, S, 0).shape == (0,)
