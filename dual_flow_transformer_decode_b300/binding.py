"""ctypes binding of libdf.so: the C-ABI entry points under the same names.

Argument marshalling only; every step of the decode path runs in the CUDA
library.  Importing this module loads the in-tree ``libdf.so`` and fails
loudly when it is missing (build it with
``python -m dual_flow_transformer_decode_b300.build``).
"""

from __future__ import annotations

import ctypes as C
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdf.so")

DF_OK, DF_ERR_ARG, DF_ERR_CUDA, DF_ERR_CAPACITY, DF_ERR_STATE, DF_ERR_TIMEOUT, DF_ERR_UNSUPPORTED, DF_ERR_DEVICE = range(8)
STATUS_NAMES = {0: "DF_OK", 1: "DF_ERR_ARG", 2: "DF_ERR_CUDA", 3: "DF_ERR_CAPACITY", 4: "DF_ERR_STATE",
                5: "DF_ERR_TIMEOUT", 6: "DF_ERR_UNSUPPORTED", 7: "DF_ERR_DEVICE"}
DF_F32, DF_BF16 = 0, 1


class df_config(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                       "ffn_hidden", "vocab", "n_experts", "top_k", "expert_hidden")] + [
        ("rope_theta", C.c_float), ("norm_eps", C.c_float), ("dtype", C.c_int),
        ("max_batch", C.c_int), ("max_len", C.c_int), ("aux_top_k", C.c_int), ("page_len", C.c_int),
        ("n_pages", C.c_int)]


class df_weights(C.Structure):
    _fields_ = [("emb1", C.c_void_p), ("emb2", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("attn_norm", C.POINTER(C.c_void_p)), ("wqkv", C.POINTER(C.c_void_p)),
                ("wo", C.POINTER(C.c_void_p)), ("mlp_norm", C.POINTER(C.c_void_p)),
                ("wgu", C.POINTER(C.c_void_p)), ("wd", C.POINTER(C.c_void_p)),
                ("router", C.POINTER(C.c_void_p)), ("a", C.POINTER(C.c_void_p)),
                ("b", C.POINTER(C.c_void_p)), ("c", C.POINTER(C.c_void_p))]


class DFError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None

EXPORTS = ["df_workspace_bytes", "df_create", "df_prefill", "df_set_length", "df_decode_step",
           "df_decode_step_host", "df_set_mode", "df_debug_outputs", "df_sync", "df_length",
           "df_step_kernels", "df_time_op", "df_last_error", "df_destroy", "df_decode_step_noalloc",
           "df_generate", "df_set_batch", "df_prefill_seq", "df_release_seq", "df_seq_lengths", "df_seq_pages",
           "df_decode_step_host_async", "df_host_wait"]

DF_OP = {"qkv": 0, "attn": 1, "wo": 2, "gateup": 3, "down": 4, "lmhead": 5, "moe": 6, "layers": 7}


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libdf.so not built at {_LIB_PATH}; run python -m dual_flow_transformer_decode_b300.build")
    L = C.CDLL(_LIB_PATH)
    vp, i, P = C.c_void_p, C.c_int, C.POINTER
    L.df_workspace_bytes.argtypes = [P(df_config), P(C.c_size_t)]
    L.df_workspace_bytes.restype = C.c_size_t
    L.df_create.argtypes = [P(df_config), P(df_weights), vp, vp, vp, P(vp)]
    L.df_create.restype = i
    L.df_prefill.argtypes = [vp, vp, i, i]
    L.df_prefill.restype = i
    L.df_set_length.argtypes = [vp, i, i]
    L.df_set_length.restype = i
    L.df_decode_step.argtypes = [vp, vp, vp, vp, vp]
    L.df_decode_step.restype = i
    L.df_decode_step_noalloc.argtypes = [vp, vp, vp, vp, vp]
    L.df_decode_step_noalloc.restype = i
    L.df_generate.argtypes = [vp, vp, i, C.c_ulonglong, vp, vp]
    L.df_generate.restype = i
    L.df_set_batch.argtypes = [vp, i]
    L.df_set_batch.restype = i
    L.df_prefill_seq.argtypes = [vp, i, vp, i]
    L.df_prefill_seq.restype = i
    L.df_release_seq.argtypes = [vp, i]
    L.df_release_seq.restype = i
    L.df_seq_lengths.argtypes = [vp, P(C.c_int32)]
    L.df_seq_lengths.restype = i
    L.df_seq_pages.argtypes = [vp, i, P(C.c_int32), i]
    L.df_seq_pages.restype = i
    L.df_decode_step_host.argtypes = [vp, vp, vp, vp, vp]
    L.df_decode_step_host.restype = i
    L.df_decode_step_host_async.argtypes = [vp, vp, vp, vp, vp]
    L.df_decode_step_host_async.restype = i
    L.df_host_wait.argtypes = [vp]
    L.df_host_wait.restype = i
    L.df_set_mode.argtypes = [vp, i, i]
    L.df_set_mode.restype = i
    L.df_debug_outputs.argtypes = [vp, vp, vp, vp, vp]
    L.df_debug_outputs.restype = i
    L.df_sync.argtypes = [vp]
    L.df_sync.restype = i
    L.df_length.argtypes = [vp]
    L.df_length.restype = i
    L.df_step_kernels.argtypes = [vp]
    L.df_step_kernels.restype = i
    L.df_time_op.argtypes = [vp, i, i, P(C.c_float)]
    L.df_time_op.restype = i
    L.df_last_error.argtypes = [vp]
    L.df_last_error.restype = C.c_char_p
    L.df_destroy.argtypes = [vp]
    L.df_destroy.restype = None
    _lib = L
    return L


def check(ctx, status: int, what: str) -> None:
    if status != DF_OK:
        msg = lib().df_last_error(ctx).decode() if ctx else ""
        raise DFError(status, f"{what}: {msg}")


def make_config(cfg, max_batch: int, max_len: int, page_len: int = 0, n_pages: int = 0) -> df_config:
    return df_config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                     cfg.ffn_hidden if not cfg.n_experts else 0, cfg.vocab, cfg.n_experts, cfg.top_k,
                     cfg.expert_hidden, float(cfg.rope_theta), float(cfg.norm_eps),
                     DF_BF16 if cfg.dtype == "bf16" else DF_F32, max_batch, max_len,
                     getattr(cfg, "aux_top_k", 0) if cfg.n_experts else 0, page_len, n_pages)


def df_workspace_bytes(c: df_config) -> tuple[int, int]:
    kv = C.c_size_t(0)
    ws = lib().df_workspace_bytes(C.byref(c), C.byref(kv))
    return int(ws), int(kv.value)


def df_create(c: df_config, w: df_weights, kv_ptr: int, ws_ptr: int, stream: int) -> int:
    ctx = C.c_void_p()
    st = lib().df_create(C.byref(c), C.byref(w), C.c_void_p(kv_ptr), C.c_void_p(ws_ptr), C.c_void_p(stream),
                         C.byref(ctx))
    if st != DF_OK:
        raise DFError(st, "df_create failed")
    return ctx.value


def df_prefill(ctx, tokens_ptr: int, B: int, n: int) -> None:
    check(ctx, lib().df_prefill(ctx, C.c_void_p(tokens_ptr), B, n), "df_prefill")


def df_set_length(ctx, B: int, t: int) -> None:
    check(ctx, lib().df_set_length(ctx, B, t), "df_set_length")


def df_decode_step(ctx, tokens_ptr: int, logp_mix_ptr: int = 0, argmax_ptr: int = 0, alpha_ptr: int = 0) -> None:
    check(ctx, lib().df_decode_step(ctx, C.c_void_p(tokens_ptr), C.c_void_p(logp_mix_ptr or None),
                                    C.c_void_p(argmax_ptr or None), C.c_void_p(alpha_ptr or None)),
          "df_decode_step")


def df_decode_step_noalloc(ctx, tokens_ptr: int, logp_mix_ptr: int = 0, argmax_ptr: int = 0,
                           alpha_ptr: int = 0) -> None:
    check(ctx, lib().df_decode_step_noalloc(ctx, C.c_void_p(tokens_ptr), C.c_void_p(logp_mix_ptr or None),
                                            C.c_void_p(argmax_ptr or None), C.c_void_p(alpha_ptr or None)),
          "df_decode_step_noalloc")


def df_generate(ctx, tokens_ptr: int, n_steps: int, seed: int, out_tokens_ptr: int, logp_mix_ptr: int = 0) -> None:
    check(ctx, lib().df_generate(ctx, C.c_void_p(tokens_ptr or None), n_steps, C.c_ulonglong(seed & (2 ** 64 - 1)),
                                 C.c_void_p(out_tokens_ptr or None), C.c_void_p(logp_mix_ptr or None)),
          "df_generate")


def df_decode_step_host(ctx, tokens_ptr: int, logp_mix_ptr: int = 0, argmax_ptr: int = 0,
                        alpha_ptr: int = 0) -> None:
    check(ctx, lib().df_decode_step_host(ctx, C.c_void_p(tokens_ptr), C.c_void_p(logp_mix_ptr or None),
                                         C.c_void_p(argmax_ptr or None), C.c_void_p(alpha_ptr or None)),
          "df_decode_step_host")


def df_set_mode(ctx, aux_on: int, ungrouped: int) -> None:
    check(ctx, lib().df_set_mode(ctx, aux_on, ungrouped), "df_set_mode")


def df_debug_outputs(ctx, logp1: int = 0, logp2: int = 0, topk: int = 0, router: int = 0) -> None:
    check(ctx, lib().df_debug_outputs(ctx, C.c_void_p(logp1 or None), C.c_void_p(logp2 or None),
                                      C.c_void_p(topk or None), C.c_void_p(router or None)), "df_debug_outputs")


def df_decode_step_host_async(ctx, tokens_ptr: int, logp_mix_ptr: int = 0, argmax_ptr: int = 0,
                              alpha_ptr: int = 0) -> None:
    check(ctx, lib().df_decode_step_host_async(ctx, C.c_void_p(tokens_ptr), C.c_void_p(logp_mix_ptr or None),
                                               C.c_void_p(argmax_ptr or None), C.c_void_p(alpha_ptr or None)),
          "df_decode_step_host_async")


def df_host_wait(ctx) -> None:
    check(ctx, lib().df_host_wait(ctx), "df_host_wait")


def df_sync(ctx) -> None:
    check(ctx, lib().df_sync(ctx), "df_sync")


def df_set_batch(ctx, B: int) -> None:
    check(ctx, lib().df_set_batch(ctx, B), "df_set_batch")


def df_prefill_seq(ctx, b: int, tokens_ptr: int, n: int) -> None:
    check(ctx, lib().df_prefill_seq(ctx, b, C.c_void_p(tokens_ptr or None), n), "df_prefill_seq")


def df_release_seq(ctx, b: int) -> None:
    check(ctx, lib().df_release_seq(ctx, b), "df_release_seq")


def df_seq_lengths(ctx, max_batch: int) -> list[int]:
    out = (C.c_int32 * max_batch)()
    check(ctx, lib().df_seq_lengths(ctx, out), "df_seq_lengths")
    return list(out)


def df_seq_pages(ctx, b: int, cap: int = 1 << 16) -> list[int]:
    out = (C.c_int32 * cap)()
    n = lib().df_seq_pages(ctx, b, out, cap)
    if n < 0:
        raise DFError(DF_ERR_ARG, "df_seq_pages: bad slot or contiguous cache")
    return list(out[:min(n, cap)])


def df_length(ctx) -> int:
    return lib().df_length(ctx)


def df_step_kernels(ctx) -> int:
    return lib().df_step_kernels(ctx)


def df_time_op(ctx, op: str, iters: int) -> float:
    ms = C.c_float(0)
    check(ctx, lib().df_time_op(ctx, DF_OP[op], iters, C.byref(ms)), "df_time_op")
    return float(ms.value)


def df_last_error(ctx) -> str:
    return lib().df_last_error(ctx).decode()


def df_destroy(ctx) -> None:
    lib().df_destroy(ctx)
