"""Batched (chunked) prefill against the token-serial prefill of the same
library, and against the oracle through the decode steps that follow.
MoE models route the chunk's rows, pack each expert's rows into 128-row
blocks and run the experts as grouped GEMMs.

The batched path runs every layer once per chunk of positions with tensor-core
GEMMs over B x C rows and a causal attention kernel over the cache; the
token-serial path (DF_SERIAL_PREFILL=1) runs one decode-shaped pass per
position.  Both compute the same causal Transformer over the primary flow
("Arquitectura Central": prefill runs the primary flow alone), with the same
quantisation points, so the caches agree to accumulation-order rounding."""

import os

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights

from parity_util import GpuRun, assert_parity, compare_steps, oracle_run

pytestmark = pytest.mark.gpu


def _serial(cfg, w, tok, **kw):
    os.environ["DF_SERIAL_PREFILL"] = "1"
    try:
        return GpuRun(cfg, w, tok, **kw)
    finally:
        del os.environ["DF_SERIAL_PREFILL"]


@pytest.mark.parametrize("name,n_prefill,batch", [
    ("t_bf16", 150, None),        # one chunk, ragged 64-position tiles
    ("t_bf16_b9", 40, None),      # batch 9: rows of one chunk not a multiple of 128
    ("t_bf16_long", 1100, None),  # batch 2: two chunks, attention across the chunk boundary
    ("t_bf16", 1, None),          # a single position
    ("t_bf16", 65, 1),            # batch 1, one position past a tile
    ("t_moe", 33, None),          # MoE: routed rows packed per expert
    ("t_moe", 300, None),         # MoE: several 128-row blocks per expert
])
def test_batched_prefill_matches_serial(name, n_prefill, batch, cuda_device):
    cfg = dfsynth.get_config(name).with_(n_prefill=n_prefill, n_steps=3)
    if batch is not None:
        cfg = cfg.with_(batch=batch)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    ser = _serial(cfg, w, tok)
    bat = GpuRun(cfg, w, tok)
    P = cfg.n_prefill
    kb, ks = bat.kv[:, :, :, :, :P].astype(np.float64), ser.kv[:, :, :, :, :P].astype(np.float64)
    d = np.abs(kb - ks)
    rel = float(np.sqrt((d ** 2).sum() / max((ks ** 2).sum(), 1e-30)))
    print(name, n_prefill, "prefill cache: max", d.max(), "relative rms", rel)
    assert d.max() < 0.05 and rel < 2.0 ** -8
    for a, b in zip(bat.steps, ser.steps):
        d1 = np.abs(a["logp1"] - b["logp1"]).max()
        dm = np.abs(a["logp_mix"] - b["logp_mix"]).max()
        print("  step max |dlogp1|", d1, "max |dlogp_mix|", dm)
        assert d1 < 5e-3 and dm < 5e-3
    bat.close()
    ser.close()


def test_batched_prefill_decode_matches_oracle(cuda_device):
    """Prefill through the batched path, then decode: the whole run against the
    fp64 oracle (which prefills token by token with a causal mask)."""
    cfg = dfsynth.get_config("t_bf16_long")
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    g = GpuRun(cfg, w, tok)
    o, outs = oracle_run(cfg, w, tok)
    rep = compare_steps(cfg, g.steps, outs)
    print(rep)
    assert_parity(cfg, rep)
    g.close()
