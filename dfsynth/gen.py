"""Counter-based seeded generators for weights, token ids and synthetic KV.

Every tensor is drawn from ``numpy.random.Generator(Philox(key=[seed, id]))``
with a fixed per-tensor id, so any single tensor can be regenerated on its own
(the oracle regenerates expert matrices on demand instead of holding 6.8e9
parameters in memory).  Matrices and embeddings are drawn N(0, std) in float32
and rounded to bf16-representable values, so the same numbers are exact both
as bf16 on the GPU and as float64 in the oracle.  Norm gains and coupling
vectors stay float32.

Tensor ids: 1 = token ids; 2/3 = E1/E2; 4 = LM head; 5 = final norm gain;
layer l: 100 + 32*l + j (j: attn_norm 0, wq 1, wk 2, wv 3, wo 4, mlp_norm 5,
wg 6, wu 7, wd 8, a 9, b 10, c 11, router 12); expert matrices
1_000_000 + 4*(4096*l + e) + {wg 0, wu 1, wd 2}; synthetic KV blocks
50_000_000 + 2*(65536*l + b) + {K 0, V 1}.
"""

from __future__ import annotations

import os
from collections import OrderedDict
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_LAYER_SLOTS = {"attn_norm": 0, "wq": 1, "wk": 2, "wv": 3, "wo": 4, "mlp_norm": 5,
                "wg": 6, "wu": 7, "wd": 8, "a": 9, "b": 10, "c": 11, "router": 12}
_EXPERT_SLOTS = {"wg": 0, "wu": 1, "wd": 2}
_GLOBAL_IDS = {"emb1": 2, "emb2": 3, "lm_head": 4, "final_norm": 5}
TOKENS_ID = 1
LENGTHS_ID = 6


def bf16_round_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), kept as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def tensor_id(key: tuple) -> int:
    if len(key) == 1:
        return _GLOBAL_IDS[key[0]]
    if len(key) == 2:
        layer, name = key
        return 100 + 32 * layer + _LAYER_SLOTS[name]
    layer, expert, name = key
    return 1_000_000 + 4 * (4096 * layer + expert) + _EXPERT_SLOTS[name]


def _rng(seed: int, tid: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed, tid]))


def tensor_shape(cfg, key: tuple) -> tuple:
    d, V = cfg.d_model, cfg.vocab
    if len(key) == 1:
        return {"emb1": (V, d), "emb2": (V, d), "lm_head": (V, d), "final_norm": (d,)}[key[0]]
    if len(key) == 2:
        name = key[1]
        F = cfg.mlp_hidden
        return {"attn_norm": (d,), "mlp_norm": (d,), "wq": (cfg.q_dim, d),
                "wk": (cfg.kv_dim, d), "wv": (cfg.kv_dim, d), "wo": (d, cfg.q_dim),
                "wg": (cfg.ffn_hidden, d), "wu": (cfg.ffn_hidden, d), "wd": (d, cfg.ffn_hidden),
                "a": (cfg.q_dim,), "b": (F,), "c": (d,), "router": (cfg.n_experts, d)}[name]
    name = key[2]
    Fe = cfg.expert_hidden
    return {"wg": (Fe, d), "wu": (Fe, d), "wd": (d, Fe)}[name]


def _kind(key: tuple) -> str:
    name = key[-1]
    if name in ("attn_norm", "mlp_norm", "final_norm"):
        return "gain"
    if name in ("a", "b", "c"):
        return "coupling"
    if name == "router":
        return "router"
    return "matrix"


def generate_tensor(cfg, seed: int, key: tuple) -> np.ndarray:
    """Draw one tensor (float32 array)."""
    shape = tensor_shape(cfg, key)
    g = _rng(seed, tensor_id(key))
    z = g.standard_normal(size=shape, dtype=np.float32)
    kind = _kind(key)
    if kind == "gain":
        return (np.float32(1.0) + np.float32(cfg.gain_std) * z).astype(np.float32)
    if kind == "coupling":
        return (np.float32(cfg.coup_std) * z).astype(np.float32)
    std = cfg.router_sigma if kind == "router" else cfg.w_std
    if key == ("lm_head",):
        std = std * cfg.lm_scale
    return bf16_round_f32(z * np.float32(std))


def all_keys(cfg) -> list:
    keys = [("emb1",), ("emb2",), ("lm_head",), ("final_norm",)]
    for l in range(cfg.n_layers):
        keys += [(l, n) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "a", "b", "c")]
        if cfg.is_moe:
            keys.append((l, "router"))
            for e in range(cfg.n_experts):
                keys += [(l, e, n) for n in ("wg", "wu", "wd")]
        else:
            keys += [(l, n) for n in ("wg", "wu", "wd")]
    return keys


class Weights:
    """Lazily generated, optionally cached mapping key -> float32 array.

    ``overrides`` replaces individual tensors (used by tests that tie E2 to E1
    or zero the couplings).  ``max_cached`` bounds the number of cached
    tensors (LRU) so that MoE experts can be regenerated on demand.
    """

    def __init__(self, cfg, seed: int = 0, overrides: dict | None = None,
                 max_cached: int | None = None):
        self.cfg = cfg
        self.seed = seed
        self.overrides = dict(overrides or {})
        self.max_cached = max_cached
        self._cache: OrderedDict = OrderedDict()

    def __getitem__(self, key: tuple) -> np.ndarray:
        if key in self.overrides:
            return self.overrides[key]
        if key in self._cache:
            self._cache.move_to_end(key)
            return self._cache[key]
        arr = generate_tensor(self.cfg, self.seed, key)
        self._cache[key] = arr
        if self.max_cached is not None:
            while len(self._cache) > self.max_cached:
                self._cache.popitem(last=False)
        return arr

    def keys(self) -> list:
        return all_keys(self.cfg)

    def prefetch(self, keys=None, threads: int | None = None) -> None:
        """Generate many tensors in a thread pool (counter-based draws make
        every tensor independent of the others; numpy's generators release the
        GIL while filling)."""
        keys = [k for k in (keys or self.keys()) if k not in self.overrides and k not in self._cache]
        if not keys:
            return
        threads = threads or min(len(keys), len(os.sched_getaffinity(0)))
        with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
            for key, arr in ex.map(lambda k: (k, generate_tensor(self.cfg, self.seed, k)), keys):
                self._cache[key] = arr


def tokens(cfg, seed: int = 0, batch: int | None = None) -> np.ndarray:
    """Token ids int32[B][max_prompt + n_steps], uniform over the vocabulary
    (max_prompt = n_prefill unless the workload's prompts are ragged)."""
    B = cfg.batch if batch is None else batch
    g = _rng(seed, TOKENS_ID)
    return g.integers(0, cfg.vocab, size=(B, cfg.max_prompt + cfg.n_steps), dtype=np.int64).astype(np.int32)


def prompt_lengths(cfg, seed: int = 0, batch: int | None = None) -> np.ndarray:
    """Prompt length of each sequence: n_prefill for every sequence, or for a
    ragged workload uniform integers in [n_prefill (1 - ragged),
    n_prefill (1 + ragged)] (seeded)."""
    B = cfg.batch if batch is None else batch
    if not cfg.ragged:
        return np.full(B, cfg.n_prefill, dtype=np.int64)
    lo = int(round(cfg.n_prefill * (1.0 - cfg.ragged)))
    g = _rng(seed, LENGTHS_ID)
    return g.integers(lo, cfg.max_prompt + 1, size=B, dtype=np.int64)


def synthetic_kv_block(cfg, seed: int, layer: int, b: int, n_pos: int, std: float = 1.0):
    """Seeded stand-in for a prefilled cache region of one sequence and layer.

    Returns (K, V), each float32[n_kv_heads][n_pos][head_dim] holding
    bf16-representable values drawn N(0, std).  Used where a workload's
    context is too long for the oracle to prefill it (32768 positions); the
    oracle and the GPU then start from the same cache contents.
    """
    out = []
    for kind in (0, 1):
        tid = 50_000_000 + 2 * (65536 * layer + b) + kind
        g = _rng(seed, tid)
        z = g.standard_normal(size=(cfg.n_kv_heads, n_pos, cfg.head_dim), dtype=np.float32)
        out.append(bf16_round_f32(z * np.float32(std)) if cfg.dtype == "bf16" else z * np.float32(std))
    return out[0], out[1]


class DeviceWeights:
    """Weights of the same shapes and distributions drawn on a CUDA device
    with torch's generator (fast set-up for timing runs; the values differ
    from ``Weights``, so these are never compared with the oracle)."""

    def __init__(self, cfg, seed: int = 0, device="cuda"):
        self.cfg = cfg
        self.seed = seed
        self.device = device

    def __getitem__(self, key: tuple):
        import torch
        shape = tensor_shape(self.cfg, key)
        g = torch.Generator(device=self.device)
        g.manual_seed(self.seed * 1_000_003 + tensor_id(key))
        z = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        kind = _kind(key)
        if kind == "gain":
            return 1.0 + self.cfg.gain_std * z
        if kind == "coupling":
            return self.cfg.coup_std * z
        std = self.cfg.router_sigma if kind == "router" else self.cfg.w_std
        if key == ("lm_head",):
            std = std * self.cfg.lm_scale
        return (z * std).to(torch.bfloat16).to(torch.float32)

    def keys(self) -> list:
        return all_keys(self.cfg)
