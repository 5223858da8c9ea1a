"""df_decode_step_noalloc: the decode step for callers that cannot allocate
device memory where they step the model (a serving loop held to a fixed
memory budget after start-up, or code building its own CUDA graph).  Its
split-attention partials live in a static device array instead of the
workspace.  The same kernels run on the same inputs, so two steps in a row
must give exactly what df_decode_step gives, bit for bit.

The cases cover each attention path: the CUDA-core split attention (fp32
models, and a bf16 model with DF_FORCE_GENERIC=1), whose partials go
through the static array; the persistent pass (DF_MK=1), whose segment
partials go there too; and the TMA attention kernel (bf16), which merges
its splits in distributed shared memory and uses none of it.

Kept in a file of its own, collected last, so a failure here comes after
every other test has run."""

import os

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights

pytestmark = pytest.mark.gpu


def _pair(cfg, env):
    """Two contexts over the same weights, created with `env` set (the path
    switches are read when a context is created), both prefilled."""
    import torch
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        ms = [DualFlowModel(cfg, w) for _ in range(2)]
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    pre = torch.from_numpy(tok[:, :cfg.n_prefill].copy()).cuda()
    for m in ms:
        m.prefill(pre)
    return ms, tok


@pytest.mark.parametrize("name,env", [
    ("t_fp32", {}),
    ("t_fp32_gqa", {}),
    ("t_bf16", {}),
    ("t_bf16", {"DF_FORCE_GENERIC": "1"}),
    ("t_bf16", {"DF_MK": "1"}),
    ("t_bf16_long", {"DF_FORCE_GENERIC": "1"}),
], ids=["t_fp32", "t_fp32_gqa", "t_bf16", "t_bf16_generic", "t_bf16_persistent", "t_bf16_long_generic"])
def test_noalloc_step_matches_decode_step(name, env, cuda_device):
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    cfg = dfsynth.get_config(name)
    (ref, st), tok = _pair(cfg, env)
    B, V = cfg.batch, cfg.vocab
    outs = []
    for m in (ref, st):
        lp = torch.zeros(B, V, device="cuda")
        am = torch.zeros(B, dtype=torch.int32, device="cuda")
        al = torch.zeros(B, device="cuda")
        outs.append((lp, am, al))
    for s in range(2):
        t = torch.from_numpy(tok[:, cfg.n_prefill + s].copy()).cuda()
        ref.decode_step(t, *outs[0])
        b.df_decode_step_noalloc(st.ctx, t.data_ptr(), outs[1][0].data_ptr(), outs[1][1].data_ptr(),
                                 outs[1][2].data_ptr())
        ref.sync()
        st.sync()
        for x, y in zip(outs[0], outs[1]):
            np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy(), err_msg=f"step {s}")
    assert st.length == ref.length == cfg.n_prefill + 2
    n = cfg.n_prefill + 2
    np.testing.assert_array_equal(ref.kv_view()[:, :, :B, :, :n].float().cpu().numpy(),
                                  st.kv_view()[:, :, :B, :, :n].float().cpu().numpy())
    ref.close()
    st.close()


def test_noalloc_step_rejects_partials_beyond_the_static_array(cuda_device):
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    # 512 sequences x 4 KV heads x at least one split x 8 query rows x 130
    # floats = 2.1e6 floats, beyond the 2^20 of the static array
    cfg = dfsynth.DFConfig("big_partials", n_layers=1, d_model=256, n_heads=16, n_kv_heads=4, head_dim=128,
                           ffn_hidden=256, vocab=256, dtype="f32", batch=512, n_prefill=60, n_steps=4)
    m = DualFlowModel(cfg, dfsynth.DeviceWeights(cfg, 0, "cuda"))
    m.set_length(cfg.batch, cfg.n_prefill)
    t = torch.zeros(cfg.batch, dtype=torch.int32, device="cuda")
    with pytest.raises(b.DFError) as e:
        b.df_decode_step_noalloc(m.ctx, t.data_ptr())
    assert e.value.status == b.DF_ERR_CAPACITY
    assert m.length == cfg.n_prefill
    m.close()
