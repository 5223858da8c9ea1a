#!/usr/bin/env python
"""Decode throughput of the grouped dual-flow step on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one df_decode_step: both flows of B sequences at one position
(embedding, every layer, LM head, mixture), teacher-forced from the seed.
The default workload is the largest single-GPU one: the 24-layer dense
model at batch 128 (256 stacked rows) with the cache prefilled to 4096
positions, where attention is bound by HBM and the projections by the
tensor cores.  The same run also times the dense ~1B model at batch 16 and
context 1023 (key "secondary").  With N > 1 (torchrun, one process per GPU)
every rank runs an independent replica of the workload: the path shards over
sequences with no exchange, so the value is the aggregate over ranks and the
scaling is weak.  Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dual-flow decode tokens/s @1xB300; achieved HBM GB/s vs roofline"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j.get("bf16_tflops", 1816.0)), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


def _bf16_sustained():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return 1400.0


class Clocks:
    """nvidia-smi sampler for the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                   "samples": len(sm)}
        return out


# Source files of each operation's kernels; an ncu figure is used only while
# these files are unchanged since the capture.
_CS = "dual_flow_transformer_decode_b300/csrc/"
_GEMM = [_CS + "tc_gemm.cu", _CS + "ptx.cuh", _CS + "common.cuh"]
OP_SOURCES = {
    "gateup": _GEMM, "down": _GEMM, "qkv": _GEMM, "wo": _GEMM, "lmhead": _GEMM,
    "attn": [_CS + "attn_fast.cu", _CS + "ptx.cuh", _CS + "common.cuh"],
    "moe": [_CS + "tc_moe.cu", _CS + "kernels_basic.cu", _CS + "ptx.cuh", _CS + "common.cuh"],
}


def sources_sha(op: str) -> str:
    import hashlib
    h = hashlib.sha1()
    for f in OP_SOURCES.get(op, []):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def captured_traffic(workload: str, op: str):
    """DRAM bytes (read + write) per launch from profiles/ncu_traffic.json, if
    that capture was taken on the current sources of the operation."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)[workload][op]
        if rec["sources_sha1"] == sources_sha(op):
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def dist_max(x: float, dist_mod=None, device="cpu") -> float:
    """A per-rank value's maximum over all ranks (a job's time is its slowest
    rank's); the identity on a single process."""
    if dist_mod is None:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, B: int, K: int, ms_total: float) -> float:
    """Whole-job throughput: each of `world` replicas decodes B sequences for
    K steps (weak scaling), timed by the slowest rank."""
    return world * B * K / (ms_total / 1e3)


def algorithmic_bytes(cfg, op: str, B: int, t: int, moe_union: float | None = None) -> float:
    """Bytes one launch of an operation must move: weights read once, KV read
    once, KV appended, logits written."""
    esz = 2 if cfg.dtype == "bf16" else 4
    d, qd, kvd, F = cfg.d_model, cfg.q_dim, cfg.kv_dim, cfg.ffn_hidden
    if op == "qkv":
        return (qd + 2 * kvd) * d * esz + 2 * B * kvd * esz
    if op == "attn":
        return 2.0 * B * kvd * (t + 1) * esz
    if op == "wo":
        return d * qd * esz
    if op == "gateup":
        return 2 * F * d * esz
    if op == "down":
        return d * F * esz
    if op == "lmhead":
        return cfg.vocab * d * esz + 2 * B * cfg.vocab * 4
    if op == "moe":
        touched = moe_union if moe_union is not None else cfg.n_experts
        return cfg.n_experts * d * esz + touched * 3 * cfg.expert_hidden * d * esz
    raise KeyError(op)


def algorithmic_flops(cfg, op: str, B: int, t: int, moe_union: float | None = None) -> float:
    """Flops one launch of an operation must do for B sequences at position
    t: every stacked row (primary and auxiliary) through each projection,
    except the auxiliary rows' Wk/Wv (the auxiliary flow writes no K/V);
    shared-KV attention of both flows' query heads over t + 1 positions."""
    d, qd, kvd, F = cfg.d_model, cfg.q_dim, cfg.kv_dim, cfg.ffn_hidden
    M = 2 * B
    if op == "qkv":
        return 2.0 * (M * qd + B * 2 * kvd) * d
    if op == "attn":
        return 8.0 * B * cfg.n_heads * cfg.head_dim * (t + 1)
    if op == "wo":
        return 2.0 * M * d * qd
    if op == "gateup":
        return 2.0 * M * 2 * F * d
    if op == "down":
        return 2.0 * M * d * F
    if op == "lmhead":
        return 2.0 * M * cfg.vocab * d
    if op == "moe":
        ka = max(cfg.aux_top_k, cfg.top_k)
        return 2.0 * M * cfg.n_experts * d + 2.0 * B * (cfg.top_k + ka) * 3 * cfg.expert_hidden * d
    raise KeyError(op)


def prefill_flops(cfg, B: int, P: int) -> float:
    """Multiply-add flops of prefilling P positions of B sequences through the
    primary flow: every weight matrix of every layer on each of the B*P rows,
    plus causal attention (scores and weighted values over positions <= p)."""
    d, qd, kvd = cfg.d_model, cfg.q_dim, cfg.kv_dim
    mlp = 3 * cfg.ffn_hidden * d if not cfg.n_experts else 3 * cfg.top_k * cfg.expert_hidden * d
    per_row = (qd + 2 * kvd) * d + d * qd + mlp
    attn = 4.0 * B * cfg.n_heads * cfg.head_dim * (P * (P + 1) / 2)
    return cfg.n_layers * (2.0 * B * P * per_row + attn)


def step_bytes(cfg, B: int, t: int, moe_union: float | None = None) -> float:
    L = cfg.n_layers
    per_layer = algorithmic_bytes(cfg, "qkv", B, t) + algorithmic_bytes(cfg, "attn", B, t) + \
        algorithmic_bytes(cfg, "wo", B, t)
    if cfg.n_experts:
        per_layer += algorithmic_bytes(cfg, "moe", B, t, moe_union)
    else:
        per_layer += algorithmic_bytes(cfg, "gateup", B, t) + algorithmic_bytes(cfg, "down", B, t)
    esz = 2 if cfg.dtype == "bf16" else 4
    return L * per_layer + cfg.vocab * cfg.d_model * esz + 2 * B * cfg.d_model * esz + B * cfg.vocab * 4


# ------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import dfsynth
    from dual_flow_transformer_decode_b300.model import DualFlowModel

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    cfg = dfsynth.get_config(args.config)
    B, P = cfg.batch, cfg.n_prefill
    K, W = args.steps, args.warmup
    span = max(cfg.n_steps, W + K)
    # per-sequence prompt lengths (all P unless the workload is ragged); the
    # decode steps of sequence b read tokens lens[b], lens[b] + 1, ...
    lens = dfsynth.prompt_lengths(cfg, args.seed + rank)
    max_len = int(lens.max()) + span
    tok = dfsynth.tokens(cfg.with_(n_steps=span), args.seed + rank)
    paged = cfg.page_len > 0
    n_pages = int(sum((int(n) + span + cfg.page_len - 1) // cfg.page_len for n in lens)) if paged else 0
    model = DualFlowModel(cfg, dfsynth.DeviceWeights(cfg, args.seed, dev), max_batch=B, max_len=max_len,
                          device=dev, page_len=cfg.page_len, n_pages=n_pages)
    tok_d = torch.from_numpy(tok).to(dev)
    P_mean = float(lens.mean())

    def prefill_all():
        if paged:
            model.set_batch(B)
            for b in range(B):
                model.prefill_seq(b, tok_d[b, :int(lens[b])].contiguous())
        else:
            model.prefill(tok_d[:, :P].contiguous())

    def reset(t=None):
        """Back to position t (default P, the end of the prompt).  Paged: every
        slot is prefilled again to its own prompt length and then decoded
        t - P steps, so each sequence stands t - P positions past its prompt."""
        if paged:
            prefill_all()
            for s in range((P if t is None else t) - P):
                step(s)
        else:
            model.set_length(B, P if t is None else t)

    prefill = None
    if args.quick:
        if paged:
            prefill_all()
        else:
            model.set_length(B, P)   # timing-only: cache contents do not change the work
    else:
        # prefill of the prompt (primary flow only), timed once with CUDA events
        model.sync()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(model.stream)
        prefill_all()
        p1.record(model.stream)
        model.sync()
        pms = p0.elapsed_time(p1)
        flop = sum(prefill_flops(cfg, 1, int(n)) for n in lens)
        bf16_peak = _bf16_sustained()  # the prefill runs for tens of milliseconds
        prefill = {"positions": P if not cfg.ragged else int(lens.sum()) // B, "batch": B, "ms": round(pms, 3),
                   "tokens_per_s": round(float(lens.sum()) / (pms / 1e3), 1),
                   "algorithmic_tflop": round(flop / 1e12, 3),
                   "achieved_tflops": round(flop / (pms / 1e3) / 1e12, 1),
                   "peak_tflops": bf16_peak, "peak_kind": "measured bf16 sustained",
                   "frac_of_bf16_peak": round(flop / (pms / 1e3) / 1e12 / bf16_peak, 4),
                   "path": "serial" if os.environ.get("DF_SERIAL_PREFILL") == "1" or cfg.dtype != "bf16" or
                   cfg.head_dim != 128 or (cfg.n_experts and (cfg.n_experts > 1024 or cfg.top_k > 16 or
                                                             cfg.expert_hidden % 64)) else "batched"}
    model.sync()
    # [span][B]: step s feeds sequence b its token at position lens[b] + s
    steps_idx = torch.from_numpy(lens[None, :] + np.arange(span)[:, None]).to(dev)
    steps_tok = torch.gather(tok_d.t(), 0, steps_idx).contiguous()
    # The step graph is cached per (token buffer, output buffers): feed each
    # step's ids through one fixed buffer, as a serving loop would.
    tok_buf = torch.empty(B, dtype=torch.int32, device=dev)
    lp = torch.empty(B, cfg.vocab, device=dev)
    am = torch.empty(B, dtype=torch.int32, device=dev)
    al = torch.empty(B, device=dev)
    stream = model.stream

    def barrier():
        if dist is not None:
            dist.barrier()

    def step(s):
        tok_buf.copy_(steps_tok[s])
        model.decode_step(tok_buf, lp, am, al)

    def timed(n_warm, n_timed):
        for s in range(n_warm):
            step(s)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(n_warm, n_warm + n_timed):
            step(s)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return e0.elapsed_time(e1)

    def max_over_ranks(x):
        return dist_max(x, dist, dev)

    # main measurement: grouped step
    clocks = Clocks(local_rank)
    clocks.start()
    ms_total = timed(W, K)
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total)
    kernels = model.step_kernels
    ms_step = ms_total / K
    tokens_s = job_tokens_per_s(world, B, K, ms_total)
    t_mid = P + W + K // 2           # mean position of the timed steps (ragged: offset from the mean prompt)
    t_mean = int(round(P_mean)) + W + K // 2
    if args.quick:
        model.close()
        return {"metric": METRIC, "value": round(tokens_s, 1), "unit": "tokens/s", "ms_per_step": round(ms_step, 4),
                "quick": True, "config": {"workload": cfg.name}, "kernels_per_step": kernels, "clocks": clk}

    # MoE: the experts a step actually reads, per layer, from the routing of
    # one step at t_mid: the union over the batch of the primary top-k sets
    # and of the auxiliary flow's own experts (when it has any)
    moe_union = moe_union_primary = None
    if cfg.n_experts:
        ka = max(cfg.aux_k, cfg.top_k)
        tk = torch.zeros(cfg.n_layers, B, ka, dtype=torch.int32, device=dev)
        model.debug_outputs(topk=tk)
        reset(t_mid)
        step(0)
        model.sync()
        tkh = tk.cpu().numpy()
        moe_union = float(np.mean([len(np.unique(tkh[l])) for l in range(cfg.n_layers)]))
        moe_union_primary = float(np.mean([len(np.unique(tkh[l, :, :cfg.top_k])) for l in range(cfg.n_layers)]))
        model.debug_outputs()

    # per-step latency distribution: an event pair around every step
    reset()
    for s in range(min(W, 3)):
        step(s)
    n_lat = min(K, 64)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_lat + 1)]
    torch.cuda.synchronize(dev)
    evs[0].record(stream)
    for i in range(n_lat):
        step(min(W, 3) + i)
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    lat = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(n_lat))
    latency = {"steps": n_lat, "p50_ms": round(lat[len(lat) // 2], 4),
               "p90_ms": round(lat[min(len(lat) - 1, (9 * len(lat)) // 10)], 4), "max_ms": round(lat[-1], 4)}

    # ablations on the same positions: two ungrouped passes, and primary-only decode
    abl = {}
    for name, aux, ung in (("ungrouped_two_pass", 1, 1), ("aux_off_standard_decode", 0, 0)):
        reset()
        model.set_mode(aux, ung)
        kk = min(K, 32)
        ms = max_over_ranks(timed(min(W, 3), kk)) / kk
        abl[name] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(world * B / (ms / 1e3), 1),
                     # two passes each read every weight and the whole cache (the
                     # auxiliary pass its own experts too); primary-only reads them once
                     "algorithmic_bytes": step_bytes(cfg, B, t_mean, moe_union_primary) +
                     step_bytes(cfg, B, t_mean, moe_union) if ung
                     else step_bytes(cfg, B, t_mean, moe_union_primary)}
    model.set_mode(1, 0)

    # generation: the same positions, each step fed the token drawn from
    # p_mix at the step before (one df_generate call for all K steps)
    gen_out = torch.empty(max(K, 3), B, dtype=torch.int32, device=dev)
    tok_buf.copy_(steps_tok[0])
    reset()
    model.generate(tok_buf, min(W, 3), args.seed, gen_out)  # warm-up (captures the step graph)
    reset()
    tok_buf.copy_(steps_tok[0])
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    model.generate(tok_buf, K, args.seed, gen_out)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    gms = max_over_ranks(g0.elapsed_time(g1)) / K
    generation = {"ms_per_step": round(gms, 4), "tokens_per_s": round(world * B / (gms / 1e3), 1),
                  "steps": K, "draw": "Gumbel-max over Philox4x64-10 noise, fed back on the device"}

    # dominant operation: time every op, cycling layers, with CUDA events
    reset(t_mid)
    step(0)
    ops = ["qkv", "attn", "wo"] + (["moe"] if cfg.n_experts else ["gateup", "down"]) + ["lmhead"]
    per_step_count = {o: (1 if o == "lmhead" else cfg.n_layers) for o in ops}
    op_ms = {}
    for o in ops:
        model.time_op(o, 2)
        op_ms[o] = model.time_op(o, max(4, 2 * cfg.n_layers) if o != "lmhead" else 8)
    shares = {o: op_ms[o] * per_step_count[o] for o in ops}
    dom = max(shares, key=shares.get)
    hbm_peak, _, peak_kind = _peaks()
    tc_peak = _bf16_sustained()   # every op is timed inside a seconds-long loop
    op_roof = {}
    for o in ops:
        by = algorithmic_bytes(cfg, o, B, t_mean + 1, moe_union)
        fl = algorithmic_flops(cfg, o, B, t_mean + 1, moe_union)
        t_hbm, t_tc = by / (hbm_peak * 1e9), fl / (tc_peak * 1e12)
        sec = op_ms[o] / 1e3
        if t_tc > t_hbm:
            op_roof[o] = {"bound": "tensor", "achieved": round(fl / sec / 1e12, 1), "peak": tc_peak,
                          "unit": "TFLOP/s", "frac": round(t_tc / sec, 4)}
        else:
            op_roof[o] = {"bound": "hbm", "achieved": round(by / sec / 1e9, 1), "peak": hbm_peak,
                          "unit": "GB/s", "frac": round(t_hbm / sec, 4)}
        op_roof[o].update({"ms_per_launch": round(op_ms[o], 5), "launches_per_step": per_step_count[o],
                           "algorithmic_bytes": by, "algorithmic_flops": fl,
                           "achieved_gbs": round(by / sec / 1e9, 1), "achieved_tflops": round(fl / sec / 1e12, 1)})
    r = op_roof[dom]
    roofline = {"kernel": dom, "bound": r["bound"], "achieved": r["achieved"], "peak": r["peak"],
                "unit": r["unit"], "frac": r["frac"],
                "traffic": captured_traffic(cfg.name, dom) if r["bound"] == "hbm" else None,
                "peak_source": peak_kind + (" bf16 sustained" if r["bound"] == "tensor" else " copy"),
                "ms_per_launch": r["ms_per_launch"], "algorithmic_bytes_per_launch": r["algorithmic_bytes"],
                "algorithmic_flops_per_launch": r["algorithmic_flops"]}
    sb = step_bytes(cfg, B, t_mean, moe_union)
    step_gbs = sb / (ms_step / 1e3) / 1e9
    # the step's roofline: its operations run one after another, each bound
    # by HBM bandwidth or by the tensor pipe, whichever it needs longer
    bound_ms = sum(per_step_count[o] * max(op_roof[o]["algorithmic_bytes"] / (hbm_peak * 1e9),
                                           op_roof[o]["algorithmic_flops"] / (tc_peak * 1e12)) for o in ops) * 1e3
    gemm_ops = [o for o in ops if o not in ("attn", "moe")]
    g_fl = sum(per_step_count[o] * op_roof[o]["algorithmic_flops"] for o in gemm_ops)
    g_ms = sum(per_step_count[o] * op_ms[o] for o in gemm_ops)
    step_roof = {"bound_ms": round(bound_ms, 4), "frac": round(bound_ms / ms_step, 4),
                 "gemm_phase": {"ops": gemm_ops, "tflop_per_step": round(g_fl / 1e12, 4), "ms_per_step": round(g_ms, 4),
                                "achieved_tflops": round(g_fl / (g_ms / 1e3) / 1e12, 1), "peak_tflops": tc_peak,
                                "frac_of_bf16_sustained": round(g_fl / (g_ms / 1e3) / 1e12 / tc_peak, 4)},
                 "attention_phase": {"ms_per_step": round(per_step_count["attn"] * op_ms["attn"], 4),
                                     "frac_of_hbm": op_roof["attn"]["frac"]}}

    # end to end through the host-buffer entry points (pinned host memory):
    # every step copies its tokens in and its log p_mix, argmax and alpha out.
    # The headline uses the pipelined call (output copies of step s overlap
    # step s + 1, two host output sets used in turn, one wait at the end of
    # the timed region); the synchronous call is reported beside it.
    h_tok = steps_tok.cpu().pin_memory()
    h_out = [(torch.empty(B, cfg.vocab).pin_memory(), torch.empty(B, dtype=torch.int32).pin_memory(),
              torch.empty(B).pin_memory()) for _ in range(2)]
    ke = min(K, span - min(W, 3))

    def host_run(pipelined: bool) -> float:
        reset()
        for s in range(min(W, 3)):
            if pipelined:
                model.decode_step_host_async(h_tok[s], *h_out[s % 2])
            else:
                model.decode_step_host(h_tok[s], *h_out[0])
        if pipelined:
            model.host_wait()
        barrier()
        t0 = time.perf_counter()
        for s in range(min(W, 3), min(W, 3) + ke):
            if pipelined:
                model.decode_step_host_async(h_tok[s], *h_out[s % 2])
            else:
                model.decode_step_host(h_tok[s], *h_out[0])
        if pipelined:
            model.host_wait()
        t1 = time.perf_counter()
        barrier()
        return max_over_ranks(t1 - t0)

    e2e_sync_s = host_run(False)
    e2e_s = host_run(True)
    e2e = {"value": round(world * B * ke / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": B * 4,
           "d2h_bytes_per_step": B * cfg.vocab * 4 + B * 4 + B * 4, "entry_point": "df_decode_step_host_async",
           "synchronous": {"entry_point": "df_decode_step_host", "value": round(world * B * ke / e2e_sync_s, 1)}}

    result = {
        "metric": METRIC, "value": round(tokens_s, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": cfg.name, "batch": B, "stacked_rows": 2 * B,
                   "context_at_first_step": P if not cfg.ragged else
                   {"min": int(lens.min()), "mean": round(P_mean, 1), "max": int(lens.max())},
                   "kv_cache": f"paged, {cfg.page_len} positions per page" if paged else "contiguous",
                   "layers": cfg.n_layers, "d_model": cfg.d_model, "vocab": cfg.vocab,
                   "experts": cfg.n_experts, "l2": "inputs larger than L2 (weights + KV per step >> 126 MB)",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu"},
        "step_hbm": {"algorithmic_bytes": sb, "achieved_gbs": round(step_gbs, 1),
                     "frac_of_measured": round(step_gbs / hbm_peak, 4), "frac_of_8tbs": round(step_gbs / 8000, 4)},
        "roofline": roofline,
        "step_roofline": step_roof,
        "ops": op_roof,
        "ops_ms_per_launch": {o: round(v, 5) for o, v in op_ms.items()},
        "step_latency": latency,
        "prefill": prefill,
        "moe_experts_read_per_layer": moe_union,
        "moe_experts_read_per_layer_primary": moe_union_primary,
        "ablation": abl,
        "generation": generation,
        "e2e": e2e,
        "gpu_launches": kernels * K if kernels >= 0 else None,
        "kernels_per_step": kernels,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, args.seed, budget_s=args.cpu_budget)
    model.close()
    del model
    torch.cuda.empty_cache()
    if world == 1 and args.secondary not in ("none", "", cfg.name):
        result["secondary"] = run_secondary(args, args.secondary, dev)
    if dist is not None:
        dist.destroy_process_group()
    return result


def run_secondary(args, name, dev):
    """The grouped step of a second workload, timed like the main one (W
    warm-up steps, K timed steps between synchronised CUDA events, inputs
    larger than L2) from a cache declared filled to the workload's context;
    the step's work does not depend on the cache contents."""
    import torch
    import dfsynth
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    cfg = dfsynth.get_config(name)
    B, P, K, W = cfg.batch, cfg.n_prefill, args.steps, args.warmup
    model = DualFlowModel(cfg, dfsynth.DeviceWeights(cfg, args.seed, dev), max_batch=B, max_len=P + W + K + 1,
                          device=dev)
    model.set_length(B, P)
    tok = torch.from_numpy(dfsynth.tokens(cfg.with_(n_steps=W + K), args.seed)[:, P:].T.copy()).to(dev)
    tok_buf = torch.empty(B, dtype=torch.int32, device=dev)
    lp = torch.empty(B, cfg.vocab, device=dev)
    am = torch.empty(B, dtype=torch.int32, device=dev)
    al = torch.empty(B, device=dev)
    for s in range(W):
        tok_buf.copy_(tok[s])
        model.decode_step(tok_buf, lp, am, al)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(model.stream)
    for s in range(W, W + K):
        tok_buf.copy_(tok[s])
        model.decode_step(tok_buf, lp, am, al)
    e1.record(model.stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / K
    hbm_peak, _, _ = _peaks()
    sb = step_bytes(cfg, B, P + W + K // 2, None)
    out = {"workload": name, "batch": B, "context_at_first_step": P, "ms_per_step": round(ms, 4),
           "tokens_per_s": round(B / (ms / 1e3), 1), "algorithmic_bytes": sb,
           "step_hbm_gbs": round(sb / (ms / 1e3) / 1e9, 1), "frac_of_measured": round(sb / (ms / 1e3) / 1e9 / hbm_peak, 4),
           "kernels_per_step": model.step_kernels, "steps": K, "warmup": W}
    model.close()
    del model
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------- oracle (CPU) arm

def _oracle_sample(cfg, seed, n_layers, extra=8):
    """Oracle for one sequence of the workload, with the cache filled to the
    workload's context from the seeded synthetic-cache generator."""
    import numpy as np
    import dfsynth
    from dfsynth.gen import Weights, synthetic_kv_block
    from oracle import Oracle
    sub = cfg.with_(n_layers=n_layers)
    w = Weights(sub, seed, max_cached=None if not sub.n_experts else 4 * sub.top_k * 3 * sub.n_layers)
    if not sub.n_experts:
        w.prefetch()
    o = Oracle(sub, w, 1, max_len=cfg.n_prefill + extra)
    for l in range(n_layers):
        K, V = synthetic_kv_block(sub, seed, l, 0, cfg.n_prefill)
        o.set_cache(0, l, K, V)
    o.set_length(cfg.n_prefill)
    toks = dfsynth.tokens(cfg, seed, batch=1)[0, cfg.n_prefill:]
    return o, toks


def cpu_baseline(cfg, seed, budget_s=30.0):
    """Oracle decode of one sequence on the host cores, scaled to tokens/s."""
    import numpy as np
    cores = len(os.sched_getaffinity(0))
    n_l = cfg.n_layers
    # size the sample: estimate one layer first
    o, toks = _oracle_sample(cfg, seed, 1)
    o.decode_step(toks[:1])
    t0 = time.perf_counter()
    o.decode_step(toks[1:2])
    per_layer = time.perf_counter() - t0
    n_l = max(1, min(cfg.n_layers, int(budget_s / max(per_layer, 1e-3) / 2)))
    o, toks = _oracle_sample(cfg, seed, n_l)
    o.decode_step(toks[:1])
    t0 = time.perf_counter()
    o.decode_step(toks[1:2])
    dt = time.perf_counter() - t0
    est_step = dt * cfg.n_layers / n_l
    return {"value": round(1.0 / est_step, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one sequence of {cfg.batch}, one decode step at position {cfg.n_prefill + 1}, "
                      f"{n_l} of {cfg.n_layers} layers (time scaled by layer count), synthetic cache"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import dfsynth
    cfg = dfsynth.get_config(args.config)
    cores = len(os.sched_getaffinity(0))
    K, W = args.steps, args.warmup
    # per-step sample: one sequence through n_l layers, sized to keep the run to a few minutes
    o, toks = _oracle_sample(cfg, args.seed, 1)
    o.decode_step(toks[:1])
    t0 = time.perf_counter()
    o.decode_step(toks[1:2])
    per_layer = time.perf_counter() - t0
    n_l = max(1, min(cfg.n_layers, int(120.0 / max(per_layer * (K + W), 1e-3))))
    o, toks = _oracle_sample(cfg, args.seed, n_l, extra=K + W + 2)
    toks_all = dfsynth.tokens(cfg.with_(n_steps=K + W + 2), args.seed, batch=1)[0, cfg.n_prefill:]
    for s in range(W):
        o.decode_step(toks_all[s:s + 1])
    t0 = time.perf_counter()
    for s in range(W, W + K):
        o.decode_step(toks_all[s:s + 1])
    dt = (time.perf_counter() - t0) / K * cfg.n_layers / n_l
    value = 1.0 / dt
    sample = (f"each step: one sequence of {cfg.batch}, one decode position, {n_l} of {cfg.n_layers} layers "
              f"(time scaled by layer count), synthetic cache at context {cfg.n_prefill}")
    return {"metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg.name, "batch": cfg.batch, "context_at_first_step": cfg.n_prefill},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--config", default="dense24l_b128")
    ap.add_argument("--secondary", default="dense1b_ctx1k",
                    help="a second workload timed in the same run (grouped step only); 'none' to skip")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--quick", action="store_true",
                    help="timing-only run for profiler captures: no prefill, no ablations, no e2e")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
