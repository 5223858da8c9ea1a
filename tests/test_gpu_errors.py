"""Host-side failure handling of the C-ABI: argument, capacity and state
errors are returned before anything is enqueued; a bad token id is caught by
the embedding kernel's bounds check, latched, reported by df_sync, and the
context stays usable."""

import numpy as np
import pytest

import dfsynth
from dfsynth.gen import Weights

pytestmark = pytest.mark.gpu


def _model(cfg, **kw):
    from dual_flow_transformer_decode_b300.model import DualFlowModel
    return DualFlowModel(cfg, Weights(cfg, 0), **kw)


def test_state_and_capacity_errors(cuda_device):
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    cfg = dfsynth.get_config("t_fp32").with_(n_prefill=4, n_steps=2)
    m = _model(cfg, max_batch=2, max_len=6)
    tok = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(b.DFError) as e:
        m.decode_step(tok)
    assert e.value.status == b.DF_ERR_STATE
    with pytest.raises(b.DFError) as e:
        m.prefill(torch.zeros(3, 4, dtype=torch.int32, device="cuda"))
    assert e.value.status == b.DF_ERR_CAPACITY
    with pytest.raises(b.DFError) as e:
        m.prefill(torch.zeros(2, 7, dtype=torch.int32, device="cuda"))
    assert e.value.status == b.DF_ERR_CAPACITY
    m.prefill(torch.zeros(2, 4, dtype=torch.int32, device="cuda"))
    m.decode_step(tok)
    m.decode_step(tok)
    assert m.length == 6
    with pytest.raises(b.DFError) as e:
        m.decode_step(tok)
    assert e.value.status == b.DF_ERR_CAPACITY
    with pytest.raises(b.DFError) as e:
        m.set_mode(2, 0)
    assert e.value.status == b.DF_ERR_ARG
    with pytest.raises(b.DFError) as e:
        m.debug_outputs(topk=tok)
    assert e.value.status == b.DF_ERR_ARG
    m.sync()
    m.close()


def test_bad_token_is_reported_and_context_recovers(cuda_device):
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    cfg = dfsynth.get_config("t_fp32")
    m = _model(cfg)
    m.prefill(torch.zeros(1, 3, dtype=torch.int32, device="cuda"))
    m.decode_step(torch.tensor([cfg.vocab + 5], dtype=torch.int32, device="cuda"))
    with pytest.raises(b.DFError) as e:
        m.sync()
    assert e.value.status == b.DF_ERR_DEVICE
    m.decode_step(torch.tensor([7], dtype=torch.int32, device="cuda"))
    m.sync()
    m.close()


def test_empty_prompt_then_decode(cuda_device):
    import torch
    cfg = dfsynth.get_config("t_fp32")
    m = _model(cfg)
    m.prefill(torch.zeros(1, 0, dtype=torch.int32, device="cuda"))
    lp = torch.zeros(1, cfg.vocab, device="cuda")
    m.decode_step(torch.tensor([3], dtype=torch.int32, device="cuda"), lp)
    m.sync()
    assert m.length == 1
    assert abs(float(lp.exp().sum()) - 1.0) < 1e-4
    m.close()
