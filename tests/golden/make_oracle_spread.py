"""Writes tests/golden/oracle_spread.json: how far the fp64 oracle moves from
itself when every value entering a bf16 rounding is perturbed by a relative
error of the size the GPU's own arithmetic makes there.

The GPU computes in fp32 where the oracle uses fp64: a dot product of
2048-8192 terms carries a relative error of about 1e-6, and the attention
weights P enter the P·V product as a bf16 pair hi + lo whose relative error
is below 2^-16 (about 1.5e-5).  At the full-size workloads the bf16
quantisation points (GEMM inputs, cache stores, attention queries) turn such
differences into rounding flips that cascade through the layers, so no
implementation that computes at fp32 precision can be expected to come
closer to the oracle than the oracle comes to itself under perturbations of
that size.  Each workload is run once unperturbed and then perturbed with
relative sizes 1e-6 and 2^-16, two noise draws each; the record keeps every
run and the largest deviations over them, from which the full-size parity
tests derive their tolerances.  MoE: a routing decision inside twice the
router-logit deviation is a near tie that either run may break; the
perturbed run then follows the unperturbed run's choice, so every (step,
token) pair stays comparable.  Only ``oracle/`` and ``dfsynth/`` are used.

    python tests/golden/make_oracle_spread.py [workload ...]
"""

from __future__ import annotations

import fcntl
import json
import os
import sys
import tempfile
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
    "dense1b_ctx1k": ([0, 5, 10, 15], 6, "prefill"),
    "dense1b_ctx32k": ([0, 3], 3, "synthetic"),
    "dense24l_b128": ([0, 42, 85, 127], 3, "synthetic"),
    "moe64e_top4": ([0, 10, 21, 31], 4, "synthetic"),
}
RUNS = [(1e-6, 5), (1e-6, 6), (2.0 ** -16, 5), (2.0 ** -16, 6)]   # (relative size, noise seed)


class Perturbed(Oracle):
    """The oracle with a relative perturbation before every bf16 rounding."""

    def __init__(self, *a, rel=1e-6, seed=5, **kw):
        super().__init__(*a, **kw)
        self._rel = rel
        self._rng = np.random.default_rng(seed)

    def q(self, x):
        x = np.asarray(x, dtype=np.float64)
        return bf16_rne(x * (1.0 + self._rel * self._rng.standard_normal(x.shape)))

    qkv = q
    qa = q


class Follow:
    """Routing hook: at a near tie (margin within twice the deviation of the
    row's router logits from the reference run) take the reference run's
    choice; elsewhere keep the run's own."""

    def __init__(self, ref_steps, top_k):
        self.ref, self.k = ref_steps, top_k
        self.step, self.followed, self.decisions = 0, 0, 0

    def __call__(self, kind, l, i, r, chosen):
        ref = self.ref[self.step]
        if kind == "primary":
            eps = float(np.abs(r - ref["router1"][l][i]).max())
            self._eps = eps
            srt = np.sort(r)[::-1]
            margin = srt[self.k - 1] - srt[self.k]
            other = ref["topk"][l, i]
        else:
            eps = 2.0 * self._eps
            S = set(int(x) for x in ref["topk"][l, i])
            rest = sorted((float(r[e]) for e in range(len(r)) if e not in S), reverse=True)
            margin = rest[len(chosen) - 1] - rest[len(chosen)]
            other = ref["topk_aux"][l, i]
        self.decisions += 1
        if margin <= 2 * eps and set(int(x) for x in other) != set(int(x) for x in chosen):
            self.followed += 1
            return np.asarray(other, dtype=np.int64)
        return chosen


def run(o, cfg, tok, sample, steps, cache, route=None):
    """Returns (per-step outputs, the K/V appended by the decode steps as
    [L][2][nb][Hkv][steps][hd])."""
    if cache == "prefill":
        o.prefill(tok[sample, :cfg.n_prefill])
    else:
        for i, b in enumerate(sample):
            for l in range(cfg.n_layers):
                K, V = synthetic_kv_block(cfg, 0, l, b, cfg.n_prefill)
                o.set_cache(i, l, K, V)
        o.set_length(cfg.n_prefill)
    outs = []
    for s in range(steps):
        if route is not None:
            route.step = s
        outs.append(o.decode_step(tok[sample, cfg.n_prefill + s], route=route))
    P = cfg.n_prefill
    kv = np.stack([np.stack([np.stack([arr[l][i][:, P:P + steps] for i in range(len(sample))])
                             for arr in (o.K, o.V)]) for l in range(cfg.n_layers)])
    return outs, kv


def main(names):
    out_path = os.path.join(HERE, "oracle_spread.json")
    for name in names:
        sample, steps, cache = CASES[name]
        cfg = dfsynth.get_config(name)
        w = Weights(cfg, 0, max_cached=None if not cfg.is_moe else 2048)
        if not cfg.is_moe:
            w.prefetch()
        tok = dfsynth.tokens(cfg, 0)
        t0 = time.time()
        a, kva = run(Oracle(cfg, w, len(sample), max_len=cfg.max_len), cfg, tok, sample, steps, cache)
        runs = []
        for rel, seed in RUNS:
            hook = Follow(a, cfg.top_k) if cfg.is_moe else None
            b, kvb = run(Perturbed(cfg, w, len(sample), max_len=cfg.max_len, rel=rel, seed=seed), cfg, tok,
                         sample, steps, cache, hook)
            dkv = np.abs(kva - kvb)
            r = {"perturbation": rel, "seed": seed,
                 "max_dlogp_mix": max(float(np.abs(x["logp_mix"] - y["logp_mix"]).max()) for x, y in zip(a, b)),
                 "max_dlogp1": max(float(np.abs(x["logp1"] - y["logp1"]).max()) for x, y in zip(a, b)),
                 "kv_max": float(dkv.max()),
                 "kv_rel_rms": float(np.sqrt((dkv ** 2).sum() / (kva ** 2).sum()))}
            if hook is not None:
                r.update({"routing_decisions": hook.decisions, "routing_followed": hook.followed})
            runs.append(r)
            print(name, r, flush=True)
        rec = {"sample": sample, "steps": steps, "cache": cache, "runs": runs,
               "seconds": round(time.time() - t0, 1)}
        for k in ("max_dlogp_mix", "max_dlogp1", "kv_max", "kv_rel_rms"):
            rec[k] = max(r[k] for r in runs)
        # several processes may write different workloads: merge under a lock
        with open(os.path.join(tempfile.gettempdir(), "oracle_spread.lock"), "w") as lk:
            fcntl.flock(lk, fcntl.LOCK_EX)
            res = json.load(open(out_path)) if os.path.exists(out_path) else {}
            res[name] = rec
            with open(out_path, "w") as f:
                json.dump(res, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or list(CASES))
