"""Workload descriptions (sizes and init scales only).

The five named workloads are the dual-flow decode workloads this library is
measured on: a tiny fp32 model, a dense ~1B bf16 model at context 1024, the
same model at context 32768, a 24-layer model at batch 128, and a 64-expert
MoE model with router replay.  The small ``t_*`` configurations are parity
cases that the fp64 oracle finishes in seconds while still spanning several
128-wide tiles and ragged tails.

Position bookkeeping: a sequence carries ``n_prefill + n_steps`` token ids.
``df_prefill`` consumes the first ``n_prefill`` (primary flow only) and decode
step ``s`` consumes id ``n_prefill + s`` at position ``t = n_prefill + s``.  For
a prompt of length P the first decode step carries the last prompt token, so
``n_prefill = P - 1`` (the auxiliary flow is active at the final prompt
position).  For "context C" workloads ``n_prefill = C`` and the first decode
id is drawn from the seed like a final prompt token.
"""

from dataclasses import dataclass, replace, asdict
import math


@dataclass(frozen=True)
class DFConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_hidden: int          # dense MLP hidden size (unused when n_experts > 0)
    vocab: int
    dtype: str               # "f32" or "bf16": storage type of weights, KV and GEMM inputs
    batch: int
    n_prefill: int
    n_steps: int
    n_experts: int = 0       # 0 = dense MLP
    top_k: int = 0
    expert_hidden: int = 0
    rope_theta: float = 1.0e4
    norm_eps: float = 1.0e-5
    w_std: float = 0.02      # matrices and embeddings
    coup_std: float = 0.1    # coupling vectors a, b, c
    gain_std: float = 0.0    # norm gains are 1 + N(0, gain_std)
    router_std: float = -1.0  # <0 means 1/sqrt(d_model)
    lm_scale: float = 1.0    # multiplies the LM-head draw (peaked-logit tests)
    aux_top_k: int = 0       # MoE auxiliary fan-out (0: the auxiliary flow replays the primary's top_k)
    page_len: int = 0        # >0: paged KV cache with pages of this many positions
    ragged: float = 0.0      # >0: prompt lengths uniform in n_prefill * [1 - ragged, 1 + ragged]

    @property
    def max_prompt(self) -> int:
        return int(round(self.n_prefill * (1.0 + self.ragged)))

    @property
    def max_len(self) -> int:
        return self.max_prompt + self.n_steps

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def is_moe(self) -> bool:
        return self.n_experts > 0

    @property
    def mlp_hidden(self) -> int:
        return self.expert_hidden if self.is_moe else self.ffn_hidden

    @property
    def aux_k(self) -> int:
        """Experts the auxiliary flow uses per token: the primary's top_k
        (replayed) plus aux_top_k - top_k chosen from its own router logits."""
        return max(self.aux_top_k, self.top_k) if self.is_moe else 0

    @property
    def router_sigma(self) -> float:
        return self.router_std if self.router_std > 0 else 1.0 / math.sqrt(self.d_model)

    def with_(self, **kw) -> "DFConfig":
        return replace(self, **kw)

    def as_dict(self) -> dict:
        return asdict(self)


WORKLOADS = {
    # Tiny dense dual-flow, fp32: prompt 16 ids -> 15 prefill positions, then 8
    # decode steps starting at the last prompt position.
    "tiny_fp32": DFConfig("tiny_fp32", n_layers=2, d_model=128, n_heads=4, n_kv_heads=4,
                          head_dim=32, ffn_hidden=512, vocab=512, dtype="f32",
                          batch=1, n_prefill=15, n_steps=8),
    # Dense ~1B, bf16: prompt 1024 -> 1023 prefill positions, 128 decode steps.
    "dense1b_ctx1k": DFConfig("dense1b_ctx1k", n_layers=16, d_model=2048, n_heads=16,
                              n_kv_heads=4, head_dim=128, ffn_hidden=8192, vocab=32000,
                              dtype="bf16", batch=16, n_prefill=1023, n_steps=128),
    # Same model, KV cache filled to 32768 positions, 64 decode steps.
    "dense1b_ctx32k": DFConfig("dense1b_ctx32k", n_layers=16, d_model=2048, n_heads=16,
                               n_kv_heads=4, head_dim=128, ffn_hidden=8192, vocab=32000,
                               dtype="bf16", batch=4, n_prefill=32768, n_steps=64),
    # 24 layers, batch 128 (256 stacked rows), context 4096, 32 decode steps.
    "dense24l_b128": DFConfig("dense24l_b128", n_layers=24, d_model=2048, n_heads=16,
                              n_kv_heads=4, head_dim=128, ffn_hidden=8192, vocab=32000,
                              dtype="bf16", batch=128, n_prefill=4096, n_steps=32),
    # MoE: 64 experts of SwiGLU hidden 1024, top-4 primary routing, router replay.
    "moe64e_top4": DFConfig("moe64e_top4", n_layers=16, d_model=2048, n_heads=16,
                            n_kv_heads=4, head_dim=128, ffn_hidden=0, vocab=32000,
                            dtype="bf16", batch=32, n_prefill=2048, n_steps=64,
                            n_experts=64, top_k=4, expert_hidden=1024),
}

# Small parity cases.  Sizes are chosen so that every GEMM spans several
# 128-row weight tiles with a ragged last tile (vocab 1000 = 7*128 + 104), the
# KV range spans several attention tiles with a ragged tail, and the stacked
# row count is not a multiple of 16.
TEST_CONFIGS = {
    "t_fp32": WORKLOADS["tiny_fp32"].with_(name="t_fp32", gain_std=0.1),
    "t_fp32_gqa": DFConfig("t_fp32_gqa", n_layers=2, d_model=96, n_heads=6, n_kv_heads=2,
                           head_dim=16, ffn_hidden=192, vocab=300, dtype="f32",
                           batch=3, n_prefill=9, n_steps=5, gain_std=0.1),
    "t_bf16": DFConfig("t_bf16", n_layers=2, d_model=384, n_heads=6, n_kv_heads=2,
                       head_dim=128, ffn_hidden=640, vocab=1000, dtype="bf16",
                       batch=3, n_prefill=150, n_steps=6, gain_std=0.1),
    "t_bf16_b9": DFConfig("t_bf16_b9", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2,
                          head_dim=128, ffn_hidden=512, vocab=777, dtype="bf16",
                          batch=9, n_prefill=40, n_steps=4, gain_std=0.1),
    # long enough that attention runs with several KV splits (a cluster merge)
    "t_bf16_long": DFConfig("t_bf16_long", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2,
                            head_dim=128, ffn_hidden=512, vocab=600, dtype="bf16",
                            batch=2, n_prefill=1100, n_steps=3, gain_std=0.1),
    # one sequence (2 stacked rows): the small projections run as the
    # CUDA-core GEMV
    "t_bf16_b1": DFConfig("t_bf16_b1", n_layers=2, d_model=384, n_heads=6, n_kv_heads=2,
                          head_dim=128, ffn_hidden=640, vocab=1000, dtype="bf16",
                          batch=1, n_prefill=70, n_steps=5, gain_std=0.1),
    # more than 128 stacked rows: the tensor-core GEMMs take their wide form
    # (one tile of up to 256 stacked rows per SM); 100 sequences give 200
    # rows (padded to 208), no K-split at this width, and a vocabulary of
    # more 128-row tiles than SMs (an LM head written straight from TMEM,
    # last tile ragged); 128 give exactly 256, and d_model 1024 gives two
    # K-splits reduced through L2
    "t_bf16_b100": DFConfig("t_bf16_b100", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2,
                            head_dim=128, ffn_hidden=512, vocab=20100, dtype="bf16",
                            batch=100, n_prefill=20, n_steps=3, gain_std=0.1),
    "t_bf16_b128": DFConfig("t_bf16_b128", n_layers=2, d_model=1024, n_heads=8, n_kv_heads=2,
                            head_dim=128, ffn_hidden=1024, vocab=1000, dtype="bf16",
                            batch=128, n_prefill=12, n_steps=3, gain_std=0.1),
    # more than 256 stacked rows: the projections take the CUDA-core path,
    # the attention grid (320 (sequence, KV head) pairs) more than one wave
    "t_bf16_b160": DFConfig("t_bf16_b160", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2,
                            head_dim=128, ffn_hidden=512, vocab=500, dtype="bf16",
                            batch=160, n_prefill=9, n_steps=2, gain_std=0.1),
    "t_moe": DFConfig("t_moe", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2,
                      head_dim=128, ffn_hidden=0, vocab=1000, dtype="bf16",
                      batch=5, n_prefill=33, n_steps=5, n_experts=8, top_k=2,
                      expert_hidden=192, gain_std=0.1),
    # independent auxiliary fan-out: 2 replayed + 2 own experts per token
    "t_moe_fan": DFConfig("t_moe_fan", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2,
                          head_dim=128, ffn_hidden=0, vocab=1000, dtype="bf16",
                          batch=5, n_prefill=33, n_steps=5, n_experts=8, top_k=2,
                          expert_hidden=192, gain_std=0.1, aux_top_k=4),
}

# Workload variants measured beside the named workloads (not parity cases).
VARIANTS = {
    # the MoE workload with the auxiliary flow using 8 experts per token
    # (4 replayed + 4 of its own): decode compute grows, prefill does not
    "moe64e_top4_aux8": WORKLOADS["moe64e_top4"].with_(name="moe64e_top4_aux8", aux_top_k=8),
    # the headline model over a paged cache (64-position pages): every
    # sequence at the same length, then a ragged batch whose prompt lengths
    # are uniform in [512, 1535] (mean ~1023, as the headline workload)
    "dense1b_paged": WORKLOADS["dense1b_ctx1k"].with_(name="dense1b_paged", page_len=64),
    "dense1b_ragged": WORKLOADS["dense1b_ctx1k"].with_(name="dense1b_ragged", page_len=64, ragged=0.5),
    # profiling cases: the same models, batches and contexts with two layers,
    # so that a counter capture holds a few GB on the device (every layer's
    # kernels have the full-size shapes; weights and caches still exceed L2)
    "dense24l_b128_2l": WORKLOADS["dense24l_b128"].with_(name="dense24l_b128_2l", n_layers=2),
    "dense1b_ctx32k_2l": WORKLOADS["dense1b_ctx32k"].with_(name="dense1b_ctx32k_2l", n_layers=2),
    "moe64e_top4_2l": WORKLOADS["moe64e_top4"].with_(name="moe64e_top4_2l", n_layers=2),
}


def get_config(name: str) -> DFConfig:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name in TEST_CONFIGS:
        return TEST_CONFIGS[name]
    if name in VARIANTS:
        return VARIANTS[name]
    raise KeyError(f"unknown config {name!r}; known: {sorted(WORKLOADS) + sorted(TEST_CONFIGS) + sorted(VARIANTS)}")
