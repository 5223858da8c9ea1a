"""CPU checks of the seeded input generators (`dfsynth`), the one module the
oracle and the CUDA path share: every tensor has a stream of its own, draws
are reproducible from the seed alone, and values follow the stated recipe
(bf16-representable matrices N(0, 0.02), couplings N(0, 0.1), gains
1 + N(0, gain_std), router N(0, 1/d), tokens uniform over the vocabulary,
ragged prompt lengths inside their range)."""

import numpy as np
import pytest
import torch

import dfsynth
from dfsynth.gen import all_keys, generate_tensor, tensor_id, bf16_round_f32, synthetic_kv_block

ALL = sorted(dfsynth.WORKLOADS) + sorted(dfsynth.TEST_CONFIGS)


@pytest.mark.parametrize("name", ALL)
def test_every_tensor_has_its_own_stream(name):
    cfg = dfsynth.get_config(name)
    keys = all_keys(cfg)
    ids = [tensor_id(k) for k in keys]
    assert len(set(ids)) == len(ids)
    # and none collides with the token, length or synthetic-cache streams
    reserved = {dfsynth.gen.TOKENS_ID, dfsynth.gen.LENGTHS_ID}
    assert not reserved & set(ids)
    assert max(ids) < 50_000_000


def test_draws_reproducible_from_the_seed_alone():
    cfg = dfsynth.get_config("t_bf16")
    for key in [("emb1",), (0, "wq"), (1, "c"), (0, "attn_norm")]:
        a = generate_tensor(cfg, 3, key)
        b = dfsynth.Weights(cfg, 3)[key]
        np.testing.assert_array_equal(a, b)
        assert not np.array_equal(a, generate_tensor(cfg, 4, key))
    np.testing.assert_array_equal(dfsynth.tokens(cfg, 5), dfsynth.tokens(cfg, 5))
    assert not np.array_equal(dfsynth.tokens(cfg, 5), dfsynth.tokens(cfg, 6))


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = (g.standard_normal(100_000) * 10.0 ** g.uniform(-30, 30, 100_000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(bf16_round_f32(x), ref)


def test_value_distributions():
    cfg = dfsynth.get_config("t_bf16")
    w = dfsynth.Weights(cfg, 0)
    m = w[(0, "wg")]
    assert np.all(m.view(np.uint32) & 0xFFFF == 0)  # bf16-representable
    assert abs(m.std() / cfg.w_std - 1) < 0.05 and abs(m.mean()) < 0.1 * cfg.w_std
    c = np.concatenate([w[(l, "c")] for l in range(cfg.n_layers)])
    assert abs(c.std() / cfg.coup_std - 1) < 0.1
    gn = np.concatenate([w[(l, "attn_norm")] for l in range(cfg.n_layers)])
    assert abs(gn.mean() - 1) < 0.02 and abs(gn.std() / cfg.gain_std - 1) < 0.15
    assert np.all(dfsynth.Weights(dfsynth.get_config("dense1b_ctx1k"), 0)[("final_norm",)] == 1.0)
    moe = dfsynth.get_config("t_moe")
    r = dfsynth.Weights(moe, 0)[(0, "router")]
    assert abs(r.std() * np.sqrt(moe.d_model) - 1) < 0.1


def test_tokens_and_prompt_lengths():
    cfg = dfsynth.get_config("t_bf16_b9")
    tok = dfsynth.tokens(cfg, 0)
    assert tok.shape == (cfg.batch, cfg.max_prompt + cfg.n_steps) and tok.dtype == np.int32
    assert tok.min() >= 0 and tok.max() < cfg.vocab
    big = dfsynth.tokens(cfg.with_(vocab=16), 0, batch=4096)
    counts = np.bincount(big.reshape(-1), minlength=16)
    expected = big.size / 16
    assert ((counts - expected) ** 2 / expected).sum() < 50  # chi-square, 15 dof
    np.testing.assert_array_equal(dfsynth.prompt_lengths(cfg, 0), np.full(cfg.batch, cfg.n_prefill))
    rag = dfsynth.get_config("dense1b_ragged")
    lens = dfsynth.prompt_lengths(rag, 0, batch=2048)
    lo = int(round(rag.n_prefill * (1 - rag.ragged)))
    assert lens.min() >= lo and lens.max() <= rag.max_prompt
    assert lens.min() < lo + 20 and lens.max() > rag.max_prompt - 20
    assert abs(lens.mean() - (lo + rag.max_prompt) / 2) < 15


def test_synthetic_cache_blocks():
    cfg = dfsynth.get_config("t_bf16")
    K, V = synthetic_kv_block(cfg, 0, 1, 2, 33)
    assert K.shape == V.shape == (cfg.n_kv_heads, 33, cfg.head_dim)
    assert np.all(K.view(np.uint32) & 0xFFFF == 0)
    K2, V2 = synthetic_kv_block(cfg, 0, 1, 2, 33)
    np.testing.assert_array_equal(K, K2)
    np.testing.assert_array_equal(V, V2)
    others = [synthetic_kv_block(cfg, 0, 0, 2, 33)[0], synthetic_kv_block(cfg, 0, 1, 3, 33)[0], V]
    for o in others:
        assert not np.array_equal(K, o)
    # values are drawn head-major, so the first head of a longer block starts
    # with the first head of the shorter one
    K3, _ = synthetic_kv_block(cfg, 0, 1, 2, 40)
    np.testing.assert_array_equal(K3[0, :33], K[0])
