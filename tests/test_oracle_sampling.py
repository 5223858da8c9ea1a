"""Pins of the oracle's sampling from p_mix (Philox4x64-10 uniforms and the
Gumbel-max draw) against published vectors, a library generator and the
distribution the draw must have."""

import math
import os

import numpy as np
import pytest

from oracle import log_softmax
from oracle.sampling import gumbel, philox4x64_10, sample, uniforms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x64_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(x, 16) for x in line.split()]
        rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


def test_philox_known_answer_vectors():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, out in rows:
        assert [int(x) for x in philox4x64_10(ctr, key)] == out


@pytest.mark.parametrize("ctr,key", [([5, 7, 9, 11], [123, 456]), ([0, 1, 2, 3], [2 ** 64 - 1, 17]),
                                     ([2 ** 64 - 1, 0, 5, 0], [1, 2])])
def test_philox_matches_numpy_philox(ctr, key):
    """numpy's Philox bit generator is Philox4x64-10 and advances its 256-bit
    counter by one before each block, so a generator started at counter c - 1
    returns the block of counter c."""
    full = sum(v << (64 * i) for i, v in enumerate(ctr)) - 1
    cm1 = np.array([(full >> (64 * i)) & (2 ** 64 - 1) for i in range(4)], dtype=np.uint64)
    g = np.random.Philox(counter=cm1, key=np.array(key, dtype=np.uint64))
    assert [int(x) for x in g.random_raw(4)] == [int(x) for x in philox4x64_10(ctr, key)]


def test_philox_vectorised_over_counters():
    j = np.arange(6, dtype=object)
    words = philox4x64_10([j, 3, 9, 0], [42, 0])
    for i in range(6):
        one = philox4x64_10([i, 3, 9, 0], [42, 0])
        assert [int(w[i]) for w in words] == [int(x) for x in one]


def test_uniform_layout_and_range():
    u = uniforms(7, 11, 2, 10)
    ctr_words = philox4x64_10([[0, 1, 2], 2, 11, 0], [7, 0])
    words = [int(ctr_words[v % 4][v // 4]) for v in range(10)]
    # word v % 4 of block v // 4; top 23 bits as an odd multiple of 2^-24
    np.testing.assert_array_equal(u, [(2 * (w >> 41) + 1) / 2 ** 24 for w in words])
    big = uniforms(1, 0, 0, 40000)
    assert big.min() > 0.0 and big.max() < 1.0
    k = big * 2 ** 24
    assert np.all(k == np.round(k)) and np.all(k % 2 == 1)
    assert abs(big.mean() - 0.5) < 4 * math.sqrt(1 / 12 / big.size)
    # float32 holds every value exactly
    np.testing.assert_array_equal(big.astype(np.float32).astype(np.float64), big)


def test_gumbel_moments():
    g = gumbel(3, 5, 0, 60000)
    euler_gamma = 0.5772156649015329
    assert abs(g.mean() - euler_gamma) < 4 * math.sqrt(math.pi ** 2 / 6 / g.size)
    assert abs(g.var() - math.pi ** 2 / 6) < 0.05


def test_noise_depends_on_every_counter_field():
    base = uniforms(5, 10, 1, 64)
    for other in (uniforms(6, 10, 1, 64), uniforms(5, 11, 1, 64), uniforms(5, 10, 2, 64)):
        assert np.mean(base == other) < 0.05


def test_gumbel_max_draws_follow_p():
    """Draws at many positions follow p (a dropped minus sign or a reversed
    argmax would not): chi-square over 4 symbols."""
    p = np.array([0.5, 0.25, 0.15, 0.10])
    logp = np.log(p)
    n = 4000
    counts = np.zeros(4)
    for t in range(n):
        x, _ = sample(logp, 99, t, 0)
        counts[x] += 1
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 16.3  # 99.9% point of chi-square with 3 degrees of freedom


def test_one_hot_mixture_always_draws_its_token():
    logp = np.full(50, -np.inf)
    logp[17] = 0.0
    for t in range(20):
        x, margin = sample(logp, 1, t, 3)
        assert x == 17 and margin == np.inf


def test_draw_is_argmax_of_perturbed_log_probs():
    rng = np.random.default_rng(0)
    logp = log_softmax(rng.normal(size=300))
    x, margin = sample(logp, 8, 4, 2)
    z = logp + gumbel(8, 4, 2, 300)
    assert x == int(np.argmax(z))
    s = np.sort(z)
    assert margin == pytest.approx(s[-1] - s[-2], abs=0)


def test_generate_feeds_each_draw_to_the_next_step():
    import dfsynth
    from dfsynth.gen import Weights
    from oracle import Oracle
    from oracle.sampling import generate
    cfg = dfsynth.get_config("t_fp32").with_(n_steps=3)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    P = cfg.n_prefill
    o1 = Oracle(cfg, w, tok.shape[0])
    o1.prefill(tok[:, :P])
    toks, margins, outs = generate(o1, tok[:, P], 3, seed=5)
    o2 = Oracle(cfg, w, tok.shape[0])
    o2.prefill(tok[:, :P])
    x = tok[:, P]
    for s in range(3):
        out = o2.decode_step(x)
        np.testing.assert_array_equal(out["logp_mix"], outs[s]["logp_mix"])
        drawn = [sample(out["logp_mix"][i], 5, P + s, i)[0] for i in range(len(x))]
        np.testing.assert_array_equal(toks[s], drawn)
        x = np.array(drawn)
    assert np.all(margins > 0)
