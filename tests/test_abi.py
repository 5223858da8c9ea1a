"""CPU checks of the C-ABI library: it loads, exports every entry point that
include/df.h declares, and sizes buffers on the host."""

import os
import re

import pytest

import dfsynth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(df_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from dual_flow_transformer_decode_b300 import build, binding
    build.build()
    return binding.lib()


def test_exports_every_declared_symbol(lib):
    decl = _declared()
    assert "df_decode_step" in decl and "df_create" in decl
    for n in decl:
        assert hasattr(lib, n), n
    from dual_flow_transformer_decode_b300 import binding
    assert sorted(binding.EXPORTS) == sorted(decl)


@pytest.mark.parametrize("name", ["tiny_fp32", "dense1b_ctx1k", "dense1b_ctx32k", "dense24l_b128", "moe64e_top4"])
def test_workspace_sizes(lib, name):
    from dual_flow_transformer_decode_b300 import binding
    cfg = dfsynth.get_config(name)
    ws, kv = binding.df_workspace_bytes(binding.make_config(cfg, cfg.batch, cfg.max_len))
    assert ws > 0
    esz = 2 if cfg.dtype == "bf16" else 4
    assert kv == cfg.n_layers * 2 * cfg.batch * cfg.n_kv_heads * cfg.max_len * cfg.head_dim * esz


def test_invalid_configs_rejected(lib):
    from dual_flow_transformer_decode_b300 import binding
    cfg = dfsynth.get_config("tiny_fp32")
    good = binding.make_config(cfg, 1, 16)
    assert binding.df_workspace_bytes(good)[0] > 0
    for field, val in [("n_heads", 3), ("head_dim", 31), ("ffn_hidden", 100), ("max_batch", 0),
                       ("dtype", 5), ("vocab", 0)]:
        c = binding.make_config(cfg, 1, 16)
        setattr(c, field, val)
        assert binding.df_workspace_bytes(c)[0] == 0, field


@pytest.mark.parametrize("page_len,n_pages", [(64, 40), (128, 7), (1024, 3)])
def test_paged_cache_size(lib, page_len, n_pages):
    """Paged cache: n_pages + 1 pages (the last a sink for free slots) of
    page_len positions for every layer, K and V, and KV head."""
    from dual_flow_transformer_decode_b300 import binding
    cfg = dfsynth.get_config("dense1b_ctx1k")
    ws, kv = binding.df_workspace_bytes(binding.make_config(cfg, cfg.batch, cfg.max_len, page_len, n_pages))
    assert ws > 0
    assert kv == cfg.n_layers * 2 * (n_pages + 1) * cfg.n_kv_heads * page_len * cfg.head_dim * 2
    # the persistent single-launch pass (contiguous caches only) reserves no
    # region here, so the paged workspace is the smaller one
    ws0, _ = binding.df_workspace_bytes(binding.make_config(cfg, cfg.batch, cfg.max_len))
    assert 0 < ws < ws0


def test_invalid_paged_configs_rejected(lib):
    from dual_flow_transformer_decode_b300 import binding
    cfg = dfsynth.get_config("t_bf16")
    assert binding.df_workspace_bytes(binding.make_config(cfg, 3, 160, 64, 9))[0] > 0
    for page_len, n_pages in [(32, 9), (96, 9), (64, 0), (0, 9), (1 << 21, 1)]:
        c = binding.make_config(cfg, 3, 160, page_len, n_pages)
        assert binding.df_workspace_bytes(c)[0] == 0, (page_len, n_pages)


def test_aux_top_k_range(lib):
    from dual_flow_transformer_decode_b300 import binding
    cfg = dfsynth.get_config("t_moe")
    for aux, ok in [(0, True), (2, True), (4, True), (8, True), (1, False), (9, False)]:
        c = binding.make_config(cfg.with_(aux_top_k=aux), 5, 40)
        assert (binding.df_workspace_bytes(c)[0] > 0) == ok, aux


def test_moe_batched_prefill_workspace(lib):
    """MoE models reserve the batched-prefill buffers (routed rows packed per
    expert): the workspace grows with the expert count and width."""
    from dual_flow_transformer_decode_b300 import binding
    cfg = dfsynth.get_config("t_moe")
    small, _ = binding.df_workspace_bytes(binding.make_config(cfg, 5, 40))
    big, _ = binding.df_workspace_bytes(binding.make_config(cfg.with_(expert_hidden=384), 5, 40))
    assert big > small > 0


def test_missing_library_fails_loudly():
    """Without libdf.so every binding call raises instead of computing
    anything another way (there is no CPU or library fallback; the model
    wrapper reaches the GPU only through these calls)."""
    import subprocess
    import sys
    code = r'''
import os
real = os.path.exists
os.path.exists = lambda p: False if str(p).endswith("libdf.so") else real(p)
import dfsynth
from dual_flow_transformer_decode_b300 import binding
cfg = dfsynth.get_config("t_fp32")
for call in (binding.lib,
             lambda: binding.df_workspace_bytes(binding.make_config(cfg, cfg.batch, cfg.max_len))):
    try:
        call()
    except ImportError as e:
        assert "libdf.so" in str(e), e
    else:
        raise SystemExit("no error without the library")
print("ok")
'''
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
