"""Writes tests/golden/oracle_spread.json: how far the fp64 oracle itself moves
when every value entering a bf16 rounding is perturbed by 1e-7 relative
(about one or two fp32 ulps, the size of the differences an fp32
implementation's summation order makes).

At the full-size workloads the bf16 quantisation points (GEMM inputs, cache
stores, attention queries) turn such last-bit differences into rounding flips
that cascade through the layers; this spread is the smallest log-probability
deviation any fp32 implementation can be expected to reach, and the
full-size parity tests derive their tolerance from it.  Only ``oracle/`` and
``dfsynth/`` are used.

    python tests/golden/make_oracle_spread.py [workload ...]
"""

from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import dfsynth  # noqa: E402
from dfsynth.gen import Weights, synthetic_kv_block  # noqa: E402
from oracle import Oracle, bf16_rne  # noqa: E402

# (workload, sampled sequences, decode steps, cache) — the full-size test cases
CASES = {
    "dense1b_ctx1k": ([0, 15], 4, "prefill"),
    "dense1b_ctx32k": ([0, 3], 3, "synthetic"),
    "dense24l_b128": ([0, 127], 2, "synthetic"),
    "moe64e_top4": ([0, 31], 3, "synthetic"),
}
REL = 1e-7


class Perturbed(Oracle):
    """The oracle with a relative perturbation before every bf16 rounding."""

    def __init__(self, *a, seed=5, **kw):
        super().__init__(*a, **kw)
        self._rng = np.random.default_rng(seed)

    def q(self, x):
        x = np.asarray(x, dtype=np.float64)
        return bf16_rne(x * (1.0 + REL * self._rng.standard_normal(x.shape)))

    qkv = q
    qa = q


def run(cls, cfg, w, tok, sample, steps, cache):
    """Returns (per-step outputs, the K/V appended by the decode steps as
    [L][2][nb][Hkv][steps][hd])."""
    o = cls(cfg, w, len(sample), max_len=cfg.max_len)
    if cache == "prefill":
        o.prefill(tok[sample, :cfg.n_prefill])
    else:
        for i, b in enumerate(sample):
            for l in range(cfg.n_layers):
                K, V = synthetic_kv_block(cfg, 0, l, b, cfg.n_prefill)
                o.set_cache(i, l, K, V)
        o.set_length(cfg.n_prefill)
    outs = [o.decode_step(tok[sample, cfg.n_prefill + s]) for s in range(steps)]
    P = cfg.n_prefill
    kv = np.stack([np.stack([np.stack([arr[l][i][:, P:P + steps] for i in range(len(sample))])
                             for arr in (o.K, o.V)]) for l in range(cfg.n_layers)])
    return outs, kv


def main(names):
    out_path = os.path.join(HERE, "oracle_spread.json")
    res = json.load(open(out_path)) if os.path.exists(out_path) else {}
    for name in names:
        sample, steps, cache = CASES[name]
        cfg = dfsynth.get_config(name)
        w = Weights(cfg, 0, max_cached=None if not cfg.is_moe else 2048)
        if not cfg.is_moe:
            w.prefetch()
        tok = dfsynth.tokens(cfg, 0)
        t0 = time.time()
        a, kva = run(Oracle, cfg, w, tok, sample, steps, cache)
        b, kvb = run(Perturbed, cfg, w, tok, sample, steps, cache)
        rec = {"sample": sample, "steps": steps, "cache": cache, "perturbation": REL}
        # the appended K/V: max |difference| and RMS(difference) / RMS(value)
        dkv = np.abs(kva - kvb)
        rec["kv_max"] = float(dkv.max())
        rec["kv_rel_rms"] = float(np.sqrt((dkv ** 2).sum() / (kva ** 2).sum()))
        if not cfg.is_moe:
            rec["max_dlogp_mix"] = max(float(np.abs(x["logp_mix"] - y["logp_mix"]).max()) for x, y in zip(a, b))
            rec["max_dlogp1"] = max(float(np.abs(x["logp1"] - y["logp1"]).max()) for x, y in zip(a, b))
        else:
            # A token whose routing differs between the two runs (a near tie
            # broken the other way) follows another computation from there on;
            # the spread is taken over the (step, token) pairs whose routing
            # agreed in every layer of every step so far.
            agree = np.ones(len(sample), dtype=bool)
            dm, d1, n_cmp, n_div = 0.0, 0.0, 0, 0
            for x, y in zip(a, b):
                same = np.array([np.array_equal(x["topk"][:, i], y["topk"][:, i]) for i in range(len(sample))])
                agree &= same
                for i in np.nonzero(agree)[0]:
                    dm = max(dm, float(np.abs(x["logp_mix"][i] - y["logp_mix"][i]).max()))
                    d1 = max(d1, float(np.abs(x["logp1"][i] - y["logp1"][i]).max()))
                    n_cmp += 1
                n_div += int((~agree).sum())
            rec.update({"max_dlogp_mix": dm, "max_dlogp1": d1, "pairs_compared": n_cmp, "pairs_diverged": n_div,
                        "max_drouter_layer0": max(float(np.abs(x["router1"][0] - y["router1"][0]).max())
                                                  for x, y in zip(a, b))})
        rec["seconds"] = round(time.time() - t0, 1)
        res[name] = rec
        print(name, rec, flush=True)
        with open(out_path, "w") as f:
            json.dump(res, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or list(CASES))
