"""Device-resident dual-flow model over the C-ABI (PyTorch for memory only).

``DualFlowModel`` lays the parameter set out in the library's documented
device layout (fused Wqkv, gate/up rows interleaved in blocks of 64),
allocates the KV cache and the workspace with torch, and calls the C entry
points.  No arithmetic of the decode step happens here.
"""

from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import binding as _b


def _interleave_gate_up(wg: torch.Tensor, wu: torch.Tensor) -> torch.Tensor:
    F, d = wg.shape
    return torch.stack([wg.reshape(F // 64, 64, d), wu.reshape(F // 64, 64, d)], dim=1).reshape(2 * F, d)


class DualFlowModel:
    """One dual-flow model instance on one GPU.

    ``weights`` maps keys (see ``dfsynth.gen``) to host numpy arrays or
    torch tensors (host or device).
    """

    def __init__(self, cfg, weights, max_batch: int | None = None, max_len: int | None = None,
                 device: str | torch.device = "cuda", stream: torch.cuda.Stream | None = None,
                 page_len: int = 0, n_pages: int = 0):
        """page_len > 0: paged KV cache of n_pages pages (per-sequence
        lengths; see prefill_seq / release_seq)."""
        self.cfg = cfg
        self.device = torch.device(device)
        self.max_batch = max_batch or cfg.batch
        self.max_len = max_len or cfg.max_len
        self.dtype = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.stream = stream or torch.cuda.current_stream(self.device)
        self._keep = []
        self.page_len, self.n_pages = page_len, n_pages
        self.c_cfg = _b.make_config(cfg, self.max_batch, self.max_len, page_len, n_pages)
        ws_bytes, kv_bytes = _b.df_workspace_bytes(self.c_cfg)
        if ws_bytes == 0:
            raise _b.DFError(_b.DF_ERR_ARG, "invalid configuration")
        self.kv = torch.zeros(kv_bytes, dtype=torch.uint8, device=self.device)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        self._upload(weights)
        self.ctx = _b.df_create(self.c_cfg, self.c_w, self.kv.data_ptr(), self.ws.data_ptr(),
                                self.stream.cuda_stream)

    # ------------------------------------------------------------- weights
    def _t(self, arr, dtype=None) -> torch.Tensor:
        t = arr if isinstance(arr, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(arr))
        return t.to(device=self.device, dtype=dtype or self.dtype)

    def _dev(self, t: torch.Tensor, dtype=None) -> torch.Tensor:
        t = self._t(t, dtype).contiguous()
        self._keep.append(t)
        return t

    def _ptrs(self, tensors) -> C.Array:
        arr = (C.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
        self._keep.append(arr)
        return arr

    def _upload(self, w) -> None:
        cfg = self.cfg
        f32 = torch.float32
        L = cfg.n_layers
        self.t_emb1 = self._dev(w[("emb1",)])
        self.t_emb2 = self._dev(w[("emb2",)])
        self.t_lm = self._dev(w[("lm_head",)])
        self.t_fn = self._dev(w[("final_norm",)], f32)
        an, mn, qkv, wo, gu, wd, rt, a, b, c = ([] for _ in range(10))
        for l in range(L):
            an.append(self._dev(w[(l, "attn_norm")], f32))
            mn.append(self._dev(w[(l, "mlp_norm")], f32))
            qkv.append(self._dev(torch.cat([self._t(w[(l, n)]) for n in ("wq", "wk", "wv")], 0)))
            wo.append(self._dev(w[(l, "wo")]))
            if cfg.n_experts:
                gu.append(self._dev(torch.stack([_interleave_gate_up(self._t(w[(l, e, "wg")]), self._t(w[(l, e, "wu")]))
                                                 for e in range(cfg.n_experts)])))
                wd.append(self._dev(torch.stack([self._t(w[(l, e, "wd")]) for e in range(cfg.n_experts)])))
                rt.append(self._dev(w[(l, "router")]))
            else:
                gu.append(self._dev(_interleave_gate_up(self._t(w[(l, "wg")]), self._t(w[(l, "wu")]))))
                wd.append(self._dev(w[(l, "wd")]))
            a.append(self._dev(w[(l, "a")], f32))
            b.append(self._dev(w[(l, "b")], f32))
            c.append(self._dev(w[(l, "c")], f32))
        self.c_w = _b.df_weights(self.t_emb1.data_ptr(), self.t_emb2.data_ptr(), self.t_fn.data_ptr(),
                                 self.t_lm.data_ptr(), self._ptrs(an), self._ptrs(qkv), self._ptrs(wo),
                                 self._ptrs(mn), self._ptrs(gu), self._ptrs(wd),
                                 self._ptrs(rt) if rt else None, self._ptrs(a), self._ptrs(b), self._ptrs(c))

    # ------------------------------------------------------------- calls
    def prefill(self, tokens: torch.Tensor) -> None:
        assert tokens.dtype == torch.int32 and tokens.is_cuda and tokens.is_contiguous()
        B, n = tokens.shape
        self._tok_keep = tokens
        _b.df_prefill(self.ctx, tokens.data_ptr(), B, n)

    def set_length(self, B: int, t: int) -> None:
        _b.df_set_length(self.ctx, B, t)

    # ------------------------------------------------------------- paged cache
    def set_batch(self, B: int) -> None:
        _b.df_set_batch(self.ctx, B)

    def prefill_seq(self, b: int, tokens: torch.Tensor) -> None:
        """Prefill slot b with its own prompt (device int32 [n])."""
        assert tokens.dtype == torch.int32 and tokens.is_cuda and tokens.is_contiguous() and tokens.dim() == 1
        self._keep_seq = getattr(self, "_keep_seq", {})
        self._keep_seq[b] = tokens
        _b.df_prefill_seq(self.ctx, b, tokens.data_ptr(), tokens.numel())

    def release_seq(self, b: int) -> None:
        _b.df_release_seq(self.ctx, b)

    def seq_lengths(self) -> list[int]:
        return _b.df_seq_lengths(self.ctx, self.max_batch)

    def seq_pages(self, b: int) -> list[int]:
        return _b.df_seq_pages(self.ctx, b)

    def decode_step(self, tokens: torch.Tensor, logp_mix: torch.Tensor | None = None,
                    argmax: torch.Tensor | None = None, alpha: torch.Tensor | None = None) -> None:
        assert tokens.dtype == torch.int32 and tokens.is_cuda
        _b.df_decode_step(self.ctx, tokens.data_ptr(), logp_mix.data_ptr() if logp_mix is not None else 0,
                          argmax.data_ptr() if argmax is not None else 0,
                          alpha.data_ptr() if alpha is not None else 0)

    def generate(self, tokens: torch.Tensor, n_steps: int, seed: int, out_tokens: torch.Tensor,
                 logp_mix: torch.Tensor | None = None) -> None:
        """n_steps decode steps, each fed the token drawn from p_mix at the
        step before (tokens feeds the first); out_tokens int32 [n_steps][B]
        receives the draws, logp_mix (optional) the last step's log p_mix."""
        assert tokens.dtype == torch.int32 and tokens.is_cuda
        assert out_tokens.dtype == torch.int32 and out_tokens.is_cuda and out_tokens.is_contiguous()
        assert out_tokens.numel() >= n_steps * tokens.numel()
        _b.df_generate(self.ctx, tokens.data_ptr(), n_steps, seed, out_tokens.data_ptr(),
                       logp_mix.data_ptr() if logp_mix is not None else 0)

    def decode_step_host(self, tokens: torch.Tensor, logp_mix: torch.Tensor | None = None,
                         argmax: torch.Tensor | None = None, alpha: torch.Tensor | None = None) -> None:
        assert tokens.dtype == torch.int32 and not tokens.is_cuda
        _b.df_decode_step_host(self.ctx, tokens.data_ptr(), logp_mix.data_ptr() if logp_mix is not None else 0,
                               argmax.data_ptr() if argmax is not None else 0,
                               alpha.data_ptr() if alpha is not None else 0)

    def decode_step_host_async(self, tokens: torch.Tensor, logp_mix: torch.Tensor | None = None,
                               argmax: torch.Tensor | None = None, alpha: torch.Tensor | None = None) -> None:
        """Pipelined host-buffer step: returns at once; the outputs are valid,
        and the buffers free, after host_wait()."""
        assert tokens.dtype == torch.int32 and not tokens.is_cuda
        _b.df_decode_step_host_async(self.ctx, tokens.data_ptr(),
                                     logp_mix.data_ptr() if logp_mix is not None else 0,
                                     argmax.data_ptr() if argmax is not None else 0,
                                     alpha.data_ptr() if alpha is not None else 0)

    def host_wait(self) -> None:
        _b.df_host_wait(self.ctx)

    def set_mode(self, aux_on: bool = True, ungrouped: bool = False) -> None:
        _b.df_set_mode(self.ctx, int(aux_on), int(ungrouped))

    def debug_outputs(self, logp1=None, logp2=None, topk=None, router=None) -> None:
        p = lambda t: t.data_ptr() if t is not None else 0
        _b.df_debug_outputs(self.ctx, p(logp1), p(logp2), p(topk), p(router))

    def sync(self) -> None:
        _b.df_sync(self.ctx)

    def time_op(self, op: str, iters: int) -> float:
        """Mean milliseconds per launch of one step operation (bench hook)."""
        return _b.df_time_op(self.ctx, op, iters)

    @property
    def length(self) -> int:
        return _b.df_length(self.ctx)

    @property
    def step_kernels(self) -> int:
        return _b.df_step_kernels(self.ctx)

    def kv_view(self) -> torch.Tensor:
        """The KV cache as [L][2][max_batch][Hkv][max_len][hd] (a view, no
        copy); paged mode: [L][2][n_pages + 1][Hkv][page_len][hd]."""
        cfg = self.cfg
        if self.page_len:
            return self.kv.view(self.dtype).view(cfg.n_layers, 2, self.n_pages + 1, cfg.n_kv_heads, self.page_len,
                                                 cfg.head_dim)
        return self.kv.view(self.dtype).view(cfg.n_layers, 2, self.max_batch, cfg.n_kv_heads, self.max_len,
                                             cfg.head_dim)

    def seq_kv(self, b: int) -> torch.Tensor:
        """Paged mode: slot b's cache gathered as [L][2][Hkv][length][hd] (a copy)."""
        kv = self.kv_view()
        n = self.seq_lengths()[b]
        pages = self.seq_pages(b)
        parts = [kv[:, :, p] for p in pages]
        if not parts:
            return kv[:, :, 0, :, :0]
        return torch.cat(parts, dim=3)[:, :, :, :n]

    def close(self) -> None:
        if getattr(self, "ctx", None):
            _b.df_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
