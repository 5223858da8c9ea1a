"""Sampling the next token from the mixture distribution (CPU oracle).

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the smoke
check and the benchmark's CPU-baseline leg use it.

Source.  The page "Resumen Técnico: Dual-Flow Transformers" (section
"Problema Central") describes decode as autoregressive token generation, and
its "Mecanismos Clave" (Objetivo de Mezcla) defines the next-token
distribution p_mix.  It does not say how a token is drawn from p_mix.
Reading taken here: one draw from p_mix itself (no temperature, no
truncation).  The token fed to the next decode step is that draw.

How a draw is made (the Gumbel-max construction, Gumbel 1954; see also
Maddison, Tarlow and Minka, "A* Sampling", 2014): with g_v independent
standard Gumbel variables,

    x = argmax_v ( log p_mix[v] + g_v )

is distributed as p_mix.  Ties go to the lowest index.  g_v = -log(-log u_v)
with u_v uniform on (0, 1).

Where the uniforms come from.  Each u_v is a function of (seed, position t,
sequence b, token v) only, so a draw does not depend on how the vocabulary is
split over threads:

* Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
  easy as 1, 2, 3", SC 2011): counter (v // 4, b, t, 0), key (seed, 0); word
  v % 4 of the output block.
* u = (2·(w >> 41) + 1) / 2^24 for the 64-bit word w: the top 23 bits, an odd
  multiple of 2^-24, so u lies strictly inside (0, 1) and is exact in fp32 and
  fp64 alike.
"""

from __future__ import annotations

import numpy as np

_MASK64 = (1 << 64) - 1
# Philox4x64 round multipliers and key increments (Salmon et al. 2011).
_PHILOX_M0 = 0xD2E7470EE14C6C93
_PHILOX_M1 = 0xCA5A826395121157
_PHILOX_W0 = 0x9E3779B97F4A7C15
_PHILOX_W1 = 0xBB67AE8584CAA73B


def philox4x64_10(counter, key):
    """The Philox4x64 bijection with 10 rounds.

    counter: four sequences of 64-bit unsigned integers, each of length n (or
    scalars); key: two of them.  Returns a list of four numpy object arrays
    (Python ints), the output words.  One round multiplies counter words 0 and
    2 by the two multipliers and mixes each product's high half with the other
    counter words and the key; the key is bumped by the increments between
    rounds."""
    c = [np.asarray(x, dtype=object) & _MASK64 for x in counter]
    k0, k1 = (np.asarray(x, dtype=object) & _MASK64 for x in key)
    for _ in range(10):
        p0 = _PHILOX_M0 * c[0]
        p1 = _PHILOX_M1 * c[2]
        hi0, lo0 = p0 >> 64, p0 & _MASK64
        hi1, lo1 = p1 >> 64, p1 & _MASK64
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = (k0 + _PHILOX_W0) & _MASK64
        k1 = (k1 + _PHILOX_W1) & _MASK64
    return c


def uniforms(seed: int, t: int, b: int, V: int) -> np.ndarray:
    """u_v for v = 0..V-1 at position t of sequence b (float64, exact)."""
    nblk = (V + 3) // 4
    j = np.arange(nblk, dtype=object)
    words = philox4x64_10([j, b, t, 0], [seed, 0])
    w = np.stack(words, axis=1).reshape(-1)[:V]
    top = np.array([int(x) >> 41 for x in w], dtype=np.float64)
    return (2.0 * top + 1.0) / 2.0 ** 24


def gumbel(seed: int, t: int, b: int, V: int) -> np.ndarray:
    """Standard Gumbel noise g_v = -log(-log u_v)."""
    return -np.log(-np.log(uniforms(seed, t, b, V)))


def sample(logp_mix: np.ndarray, seed: int, t: int, b: int):
    """One draw from p_mix for sequence b at position t.

    Returns (token, margin): the argmax of log p_mix + g (lowest index on
    ties) and the gap between the largest and second-largest perturbed value
    (the decision's distance from a tie)."""
    z = np.asarray(logp_mix, dtype=np.float64) + gumbel(seed, t, b, logp_mix.shape[-1])
    x = int(np.argmax(z))
    if z.shape[0] < 2:
        return x, np.inf
    top2 = np.partition(z, -2)[-2:]
    return x, float(top2[1] - top2[0])


def generate(oracle, first_tokens, n_steps: int, seed: int, seq_ids=None, aux: bool = True):
    """n_steps decode steps of `oracle` (an Oracle after its prefill), each
    fed the token drawn at the step before; the first step is fed
    first_tokens.  The draw of sequence i at the step that processes position
    t uses the noise of (seed, t, seq_ids[i]) (default: i).

    Returns (tokens [n_steps][nb], margins [n_steps][nb], outs): the token
    drawn at each step, its distance from a tie, and each step's outputs."""
    nb = len(first_tokens)
    ids = list(range(nb)) if seq_ids is None else list(seq_ids)
    tok = np.asarray(first_tokens, dtype=np.int64).copy()
    toks = np.zeros((n_steps, nb), dtype=np.int64)
    margins = np.zeros((n_steps, nb))
    outs = []
    for s in range(n_steps):
        t = oracle.t
        out = oracle.decode_step(tok, aux=aux)
        lp = out["logp_mix"] if aux else out["logp1"]
        for i in range(nb):
            toks[s, i], margins[s, i] = sample(lp[i], seed, t, ids[i])
        outs.append(out)
        tok = toks[s].copy()
    return toks, margins, outs
