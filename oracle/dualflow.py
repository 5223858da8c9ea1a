"""fp64 CPU oracle of the Dual-Flow Transformer prefill and decode step.

TEST INFRASTRUCTURE.  Plain, slow and written to be checked by eye against
the description of the method.  It shares no code with the CUDA library.

Sources.  Citations name the page "Resumen Técnico: Dual-Flow Transformers"
(gist.science, Spanish technical summary of arXiv 2608.12385) and its section
headings; its Arabic and Chinese translations on gist.science carry the same
sections.  The pages give no equations beyond the mixture formula, so every
step below that the pages leave open follows one stated reading:

* block: pre-norm LLaMA-style decoder (the results section names a "Dense
  LLaMA" model family): RMSNorm with eps 1e-5, rotate-half RoPE (theta 1e4),
  grouped-query attention (query head h reads KV head h // G), SwiGLU MLP,
  untied LM head, one final norm shared by both flows;
* coupling ("Mecanismos Clave", Acoplamiento Ligero: query level, MLP
  intermediate, MLP output):  Q2 = Wq·u2 + a ⊙ q1 with q1 the primary's
  pre-RoPE query of the same layer and position;  z2 = silu(Wg·u2) ⊙ (Wu·u2)
  + b ⊙ z1 on the post-gating product;  y2 = Wd·z2 + c ⊙ y1 before the
  residual add;
* the auxiliary flow attends to the primary K/V at positions 0..t inclusive
  and keeps no state across positions (it starts from E2[x_t] every step);
* mixture ("Mecanismos Clave", Objetivo de Mezcla): alpha = 0.5 + 0.5·Σ p1²;
* MoE ("Mecanismos Clave", Replay de Router): the router reads the normed
  residual unrounded; the primary takes the top-k logits (descending, ties to
  the lower index); each flow's gates are the softmax of its own router
  logits over that set; one b of the expert hidden size is shared by all
  experts of a layer; no capacity limit;
* independent auxiliary fan-out ("Contribuciones Clave" 3 and "Significado y
  Reivindicaciones": each flow's expert fan-out is configurable): with
  aux_top_k = k_a > k the auxiliary flow keeps the replayed set S and adds
  the k_a - k largest of its own router logits among the experts outside S
  (ties to the lower index); its gates are the softmax of its router logits
  over S followed by those extra experts; the b coupling applies to the
  replayed experts only (the primary computed no hidden state for the
  others).

Quantisation points (mirrored by the GPU): in bf16 models the GEMM inputs,
the KV-cache stores and the attention queries are rounded to bf16
(round-to-nearest-even, directly from fp64 here); everything else is fp64.
In fp32 models these roundings are the identity.

parity unpinned: the whole-step numerics have no published numbers to pin
to; each part is pinned in the tests to closed forms, special cases and
library routines instead.
"""

from __future__ import annotations

import math
from collections import OrderedDict

import numpy as np


# --------------------------------------------------------------------------
# elementwise pieces
# --------------------------------------------------------------------------

def bf16_rne(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even (one rounding).

    bf16 keeps 8 significant bits and the fp32 exponent range, so a value in
    [2^(e-1), 2^e) has quantum 2^(e-8); below the normal range the quantum is
    fixed at 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    e = np.maximum(e, -125)
    scale = np.ldexp(1.0, 8 - e)
    return np.rint(x * scale) / scale


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def silu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of head vectors x[..., hd] at positions pos.

    Pair (i, i + hd/2) is rotated by angle pos * theta^(-2i/hd).  ``pos`` is a
    scalar or broadcasts against x[..., 0].
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def log_softmax(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    return z - m - np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True))


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q·K^T / sqrt(hd)) · V for every query head.

    q: [Hq][hd] (already rotated), K, V: [Hkv][n][hd].  Query head h reads
    KV head h // (Hq/Hkv).  Returns o[Hq][hd].
    """
    Hq, hd = q.shape
    Hkv = K.shape[0]
    G = Hq // Hkv
    o = np.empty((Hq, hd), dtype=np.float64)
    for h in range(Hq):
        Kh = np.asarray(K[h // G], dtype=np.float64)
        Vh = np.asarray(V[h // G], dtype=np.float64)
        s = Kh @ q[h] / math.sqrt(hd)
        p = np.exp(s - s.max())
        p /= p.sum()
        o[h] = p @ Vh
    return o


def mixture(logp1: np.ndarray, logp2: np.ndarray):
    """p_mix = alpha·p1 + (1-alpha)·p2 with alpha = 0.5 + 0.5·Σ p1^2.

    Returns (log p_mix, alpha).  When alpha == 1 the auxiliary term vanishes.
    """
    p1 = np.exp(logp1)
    coll = float(np.sum(p1 * p1))
    alpha = 0.5 + 0.5 * coll
    la = math.log(alpha)
    if alpha >= 1.0:
        return logp1 + la, alpha
    lb = math.log1p(-alpha)
    return np.logaddexp(la + logp1, lb + logp2), alpha


def topk_desc(r: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values, in descending value order; equal values
    are ordered by ascending index."""
    order = sorted(range(len(r)), key=lambda i: (-float(r[i]), i))
    return np.array(order[:k], dtype=np.int64)


# --------------------------------------------------------------------------
# the model
# --------------------------------------------------------------------------

class Oracle:
    """Dual-flow model over ``nb`` sequences with a primary-only KV cache.

    ``weights`` maps keys (see ``dfsynth.gen``) to float32 arrays; this class
    keeps fp64 copies of the dense matrices and an LRU of expert matrices.
    The KV cache stores quantised values (bf16 values in bf16 models) as
    float64: ``K[l][s]`` and ``V[l][s]`` are [Hkv][max_len][hd].
    """

    def __init__(self, cfg, weights, nb: int, max_len: int | None = None,
                 expert_cache: int = 96):
        self.cfg = cfg
        self.w = weights
        self.nb = nb
        self.max_len = cfg.max_len if max_len is None else max_len
        self.bf16 = cfg.dtype == "bf16"
        self._w64: dict = {}
        self._exp64: OrderedDict = OrderedDict()
        self._expert_cache = expert_cache
        shape = (cfg.n_kv_heads, self.max_len, cfg.head_dim)
        self.K = [[np.zeros(shape) for _ in range(nb)] for _ in range(cfg.n_layers)]
        self.V = [[np.zeros(shape) for _ in range(nb)] for _ in range(cfg.n_layers)]
        self.t = 0

    # quantisation points -------------------------------------------------
    def q(self, x):
        """GEMM activation input."""
        return bf16_rne(x) if self.bf16 else np.asarray(x, dtype=np.float64)

    qkv = q   # KV-cache store
    qa = q    # query entering attention

    # weights ---------------------------------------------------------------
    def W(self, *key) -> np.ndarray:
        if key not in self._w64:
            self._w64[key] = np.asarray(self.w[key], dtype=np.float64)
        return self._w64[key]

    def EW(self, layer, expert, name) -> np.ndarray:
        key = (layer, expert, name)
        if key in self._exp64:
            self._exp64.move_to_end(key)
            return self._exp64[key]
        arr = np.asarray(self.w[key], dtype=np.float64)
        self._exp64[key] = arr
        while len(self._exp64) > self._expert_cache:
            self._exp64.popitem(last=False)
        return arr

    # cache -----------------------------------------------------------------
    def set_cache(self, seq: int, layer: int, K: np.ndarray, V: np.ndarray) -> None:
        """Load cache contents for positions 0..n-1 of one sequence and layer."""
        n = K.shape[1]
        self.K[layer][seq][:, :n] = self.qkv(K)
        self.V[layer][seq][:, :n] = self.qkv(V)

    def set_length(self, t: int) -> None:
        self.t = t

    # pieces of one block -----------------------------------------------------
    def _heads(self, x, nh):
        return x.reshape(x.shape[:-1] + (nh, self.cfg.head_dim))

    def _mlp_dense(self, l, u):
        """SwiGLU hidden (fp64, before rounding) for rows u[n][d]."""
        return silu(u @ self.W(l, "wg").T) * (u @ self.W(l, "wu").T)

    def _expert_hidden(self, l, e, u):
        return silu(u @ self.EW(l, e, "wg").T) * (u @ self.EW(l, e, "wu").T)

    @staticmethod
    def _aux_extra(r2: np.ndarray, S: np.ndarray, nx: int) -> np.ndarray:
        """The auxiliary flow's own nx experts: its largest router logits among
        the experts outside the replayed set S (descending, ties to the lower
        index)."""
        if nx <= 0:
            return np.zeros(0, dtype=np.int64)
        rest = [e for e in range(len(r2)) if e not in set(int(x) for x in S)]
        order = sorted(rest, key=lambda e: (-float(r2[e]), e))
        return np.array(order[:nx], dtype=np.int64)

    @staticmethod
    def _aux_extra_margin(r2: np.ndarray, S: np.ndarray, nx: int) -> float:
        """Gap between the last chosen and the first unchosen of those logits."""
        rest = sorted((float(r2[e]) for e in range(len(r2)) if e not in set(int(x) for x in S)), reverse=True)
        return rest[nx - 1] - rest[nx] if len(rest) > nx else np.inf

    def _router(self, l, h):
        cfg = self.cfg
        return rmsnorm(h, self.W(l, "mlp_norm"), cfg.norm_eps) @ self.W(l, "router").T

    # prefill -------------------------------------------------------------------
    def prefill(self, tok: np.ndarray) -> None:
        """Primary flow alone over positions 0..n-1 of every sequence
        ("Arquitectura Central": the primary flow processes the whole prompt and
        writes the persistent KV cache; the auxiliary flow is skipped).

        This is the standard causal Transformer over the whole prompt, written
        with a causal mask rather than position by position.
        """
        cfg = self.cfg
        tok = np.asarray(tok)
        n = tok.shape[1]
        pos = np.arange(n)
        mask = np.tril(np.ones((n, n), dtype=bool))
        G = cfg.group
        for s in range(self.nb):
            h = self.W("emb1")[tok[s]].copy()
            for l in range(cfg.n_layers):
                u = self.q(rmsnorm(h, self.W(l, "attn_norm"), cfg.norm_eps))
                qf = self._heads(u @ self.W(l, "wq").T, cfg.n_heads)       # [n][Hq][hd]
                kf = self._heads(u @ self.W(l, "wk").T, cfg.n_kv_heads)
                vf = self._heads(u @ self.W(l, "wv").T, cfg.n_kv_heads)
                kr = self.qkv(rope(kf, pos[:, None], cfg.rope_theta))
                self.K[l][s][:, :n] = kr.transpose(1, 0, 2)
                self.V[l][s][:, :n] = self.qkv(vf).transpose(1, 0, 2)
                qr = self.qa(rope(qf, pos[:, None], cfg.rope_theta))
                o = np.empty((n, cfg.n_heads, cfg.head_dim))
                for hh in range(cfg.n_heads):
                    Kh = self.K[l][s][hh // G, :n]
                    Vh = self.V[l][s][hh // G, :n]
                    sc = qr[:, hh] @ Kh.T / math.sqrt(cfg.head_dim)
                    sc = np.where(mask, sc, -np.inf)
                    p = np.exp(sc - sc.max(axis=1, keepdims=True))
                    p /= p.sum(axis=1, keepdims=True)
                    o[:, hh] = p @ Vh
                h = h + self.q(o.reshape(n, -1)) @ self.W(l, "wo").T
                if cfg.is_moe:
                    y, _, _ = self._moe_rows(l, h)
                else:
                    u2 = self.q(rmsnorm(h, self.W(l, "mlp_norm"), cfg.norm_eps))
                    y = self.q(self._mlp_dense(l, u2)) @ self.W(l, "wd").T
                h = h + y
        self.t = n

    def _moe_rows(self, l, h):
        """MoE MLP for primary rows h[n][d] with their own routing (prefill)."""
        cfg = self.cfg
        r = self._router(l, h)
        u2 = self.q(rmsnorm(h, self.W(l, "mlp_norm"), cfg.norm_eps))
        y = np.zeros_like(h)
        sets = []
        for i in range(h.shape[0]):
            S = topk_desc(r[i], cfg.top_k)
            g = np.exp(log_softmax(r[i][S]))
            for j, e in enumerate(S):
                z = self._expert_hidden(l, e, u2[i:i + 1])
                y[i] += g[j] * (self.q(z) @ self.EW(l, e, "wd").T)[0]
            sets.append(S)
        return y, sets, r

    # decode ----------------------------------------------------------------------
    def decode_step(self, tok: np.ndarray, aux: bool = True, trace: bool = False, route=None) -> dict:
        """One decode position t for every sequence.

        Primary ("Arquitectura Central", Flujo Primario): a standard causal step
        that appends K/V at t.  Auxiliary (Flujo Auxiliar, only at the final
        prompt position and later): starts from E2[x_t], couples to the
        primary through a, b, c, attends to the primary K/V 0..t, writes
        nothing.  Output: the mixture of the two next-token distributions
        ("Mecanismos Clave", Objetivo de Mezcla).

        route: optional comparison hook for MoE models,
        route(kind, layer, seq, logits, chosen) -> experts to use, called
        after each routing decision with kind "primary" (the top-k set S) or
        "aux" (the auxiliary flow's own extra experts).  It lets a comparison
        follow another implementation through a decision that is a tie at
        that implementation's precision; the returned set replaces the
        chosen one in that step's arithmetic, which is otherwise unchanged.
        The returned indices are recorded in the outputs ("topk",
        "topk_aux").
        """
        cfg = self.cfg
        tok = np.asarray(tok).reshape(-1)
        t = self.t
        if t >= self.max_len:
            raise ValueError("cache full")
        G = cfg.group
        L = cfg.n_layers
        out = {"t": t}

        # ---- primary flow: the whole step, all layers ----
        h1 = self.W("emb1")[tok].copy()                      # [nb][d]
        saved = []
        topk_sets = np.zeros((L, self.nb, max(cfg.top_k, 1)), dtype=np.int64)
        topk_margin = np.full((L, self.nb), np.inf)
        router_logits = []
        ptrace = []
        for l in range(L):
            u = self.q(rmsnorm(h1, self.W(l, "attn_norm"), cfg.norm_eps))
            q1 = u @ self.W(l, "wq").T                          # pre-RoPE, fp64
            k1 = self._heads(u @ self.W(l, "wk").T, cfg.n_kv_heads)
            v1 = self._heads(u @ self.W(l, "wv").T, cfg.n_kv_heads)
            o1 = np.empty((self.nb, cfg.q_dim))
            for s in range(self.nb):
                self.K[l][s][:, t] = self.qkv(rope(k1[s], t, cfg.rope_theta))
                self.V[l][s][:, t] = self.qkv(v1[s])
                qr = self.qa(rope(self._heads(q1[s], cfg.n_heads), t, cfg.rope_theta))
                o1[s] = attend(qr, self.K[l][s][:, :t + 1], self.V[l][s][:, :t + 1]).reshape(-1)
            h1 = h1 + self.q(o1) @ self.W(l, "wo").T
            if trace:
                ptrace.append({"h1_attn": h1.copy()})
            if cfg.is_moe:
                r1 = self._router(l, h1)
                u2 = self.q(rmsnorm(h1, self.W(l, "mlp_norm"), cfg.norm_eps))
                y1 = np.zeros_like(h1)
                z1 = {}
                sets = []
                for s in range(self.nb):
                    S = topk_desc(r1[s], cfg.top_k)
                    if route is not None:
                        S = np.asarray(route("primary", l, s, r1[s], S), dtype=np.int64)
                    sets.append(S)
                    topk_sets[l, s] = S
                    if cfg.n_experts > cfg.top_k:
                        srt = np.sort(r1[s])[::-1]
                        topk_margin[l, s] = srt[cfg.top_k - 1] - srt[cfg.top_k]
                    g1 = np.exp(log_softmax(r1[s][S]))
                    for j, e in enumerate(S):
                        z = self._expert_hidden(l, e, u2[s:s + 1])[0]
                        z1[(s, j)] = z
                        y1[s] += g1[j] * (self.q(z) @ self.EW(l, e, "wd").T)
                router_logits.append(r1)
                saved.append({"q1": q1, "z1": z1, "y1": y1, "sets": sets})
            else:
                u2 = self.q(rmsnorm(h1, self.W(l, "mlp_norm"), cfg.norm_eps))
                z1 = self._mlp_dense(l, u2)
                y1 = self.q(z1) @ self.W(l, "wd").T
                saved.append({"q1": q1, "z1": z1, "y1": y1})
            h1 = h1 + y1
        logits1 = self.q(rmsnorm(h1, self.W("final_norm"), cfg.norm_eps)) @ self.W("lm_head").T
        logp1 = log_softmax(logits1)
        out["logits1"] = logits1
        out["logp1"] = logp1
        out["argmax1"] = np.argmax(logp1, axis=1)
        out["topk"] = topk_sets
        out["topk_margin"] = topk_margin
        if cfg.is_moe:
            out["router1"] = np.stack(router_logits)

        if aux:
            # ---- auxiliary flow: reads the primary cache and saved state ----
            h2 = self.W("emb2")[tok].copy()
            nxa = max(cfg.aux_k - cfg.top_k, 0) if cfg.is_moe else 0
            aux_extra = np.zeros((L, self.nb, nxa), dtype=np.int64)
            aux_margin = np.full((L, self.nb), np.inf)
            router2 = []
            tr = []
            for l in range(L):
                sv = saved[l]
                u = self.q(rmsnorm(h2, self.W(l, "attn_norm"), cfg.norm_eps))
                Q2 = u @ self.W(l, "wq").T + self.W(l, "a") * sv["q1"]
                o2 = np.empty((self.nb, cfg.q_dim))
                for s in range(self.nb):
                    qr = self.qa(rope(self._heads(Q2[s], cfg.n_heads), t, cfg.rope_theta))
                    o2[s] = attend(qr, self.K[l][s][:, :t + 1], self.V[l][s][:, :t + 1]).reshape(-1)
                h2 = h2 + self.q(o2) @ self.W(l, "wo").T
                h2_attn = h2.copy()
                if cfg.is_moe:
                    r2 = self._router(l, h2)
                    router2.append(r2)
                    u2 = self.q(rmsnorm(h2, self.W(l, "mlp_norm"), cfg.norm_eps))
                    y2 = np.zeros_like(h2)
                    nx = cfg.aux_k - cfg.top_k
                    for s in range(self.nb):
                        S = sv["sets"][s]
                        X = self._aux_extra(r2[s], S, nx)
                        if route is not None and nx > 0:
                            X = np.asarray(route("aux", l, s, r2[s], X), dtype=np.int64)
                        aux_extra[l, s] = X
                        if nx > 0:
                            aux_margin[l, s] = self._aux_extra_margin(r2[s], S, nx)
                        SA = np.concatenate([S, X]).astype(np.int64)
                        g2 = np.exp(log_softmax(r2[s][SA]))
                        for j, e in enumerate(SA):
                            z = self._expert_hidden(l, e, u2[s:s + 1])[0]
                            if j < len(S):
                                z = z + self.W(l, "b") * sv["z1"][(s, j)]
                            y2[s] += g2[j] * (self.q(z) @ self.EW(l, e, "wd").T)
                    y2 = y2 + self.W(l, "c") * sv["y1"]
                else:
                    u2 = self.q(rmsnorm(h2, self.W(l, "mlp_norm"), cfg.norm_eps))
                    z2 = self._mlp_dense(l, u2) + self.W(l, "b") * sv["z1"]
                    y2 = self.q(z2) @ self.W(l, "wd").T + self.W(l, "c") * sv["y1"]
                h2 = h2 + y2
                if trace:
                    tr.append({"h2_attn": h2_attn, "h2": h2.copy(), "Q2": Q2, "o2": o2})
            logits2 = self.q(rmsnorm(h2, self.W("final_norm"), cfg.norm_eps)) @ self.W("lm_head").T
            logp2 = log_softmax(logits2)
            mix = np.empty_like(logp1)
            alpha = np.empty(self.nb)
            for s in range(self.nb):
                mix[s], alpha[s] = mixture(logp1[s], logp2[s])
            out["logits2"] = logits2
            out["logp2"] = logp2
            if cfg.is_moe:
                out["topk_aux"] = aux_extra
                out["topk_aux_margin"] = aux_margin
                out["router2"] = np.stack(router2)
            out["logp_mix"] = mix
            out["alpha"] = alpha
            out["argmax"] = np.argmax(mix, axis=1)
            srt = np.sort(mix, axis=1)
            out["argmax_margin"] = srt[:, -1] - srt[:, -2]
            if trace:
                out["trace"] = tr
                out["trace_primary"] = ptrace
        srt1 = np.sort(logp1, axis=1)
        out["argmax1_margin"] = srt1[:, -1] - srt1[:, -2]
        self.t = t + 1
        return out
