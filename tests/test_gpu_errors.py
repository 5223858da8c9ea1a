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


def test_slot_calls_need_a_paged_cache(cuda_device):
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    cfg = dfsynth.get_config("t_bf16")
    m = _model(cfg)
    m.prefill(torch.zeros(cfg.batch, 5, dtype=torch.int32, device="cuda"))
    for call in (lambda: m.set_batch(2), lambda: m.release_seq(0),
                 lambda: m.prefill_seq(0, torch.zeros(3, dtype=torch.int32, device="cuda"))):
        with pytest.raises(b.DFError) as e:
            call()
        assert e.value.status == b.DF_ERR_UNSUPPORTED
    with pytest.raises(b.DFError):
        m.seq_pages(0)
    assert m.seq_lengths()[:cfg.batch] == [5] * cfg.batch
    m.sync()
    m.close()


def test_paged_and_generation_argument_errors(cuda_device):
    """Every refusal comes back before anything is enqueued: the lengths and
    the page pool are unchanged and the next valid call works."""
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    cfg = dfsynth.get_config("t_bf16")
    m = _model(cfg, max_batch=3, max_len=100, page_len=64, n_pages=4)
    tok = torch.zeros(40, dtype=torch.int32, device="cuda")
    with pytest.raises(b.DFError) as e:
        m.prefill_seq(0, tok)          # before any batch size is set
    assert e.value.status == b.DF_ERR_STATE
    m.set_batch(2)
    with pytest.raises(b.DFError) as e:
        m.prefill_seq(2, tok)          # slot beyond the batch
    assert e.value.status == b.DF_ERR_ARG
    with pytest.raises(b.DFError) as e:
        m.prefill_seq(0, torch.zeros(101, dtype=torch.int32, device="cuda"))
    assert e.value.status == b.DF_ERR_CAPACITY
    with pytest.raises(b.DFError) as e:
        m.set_batch(4)                 # more slots than max_batch
    assert e.value.status == b.DF_ERR_ARG
    m.prefill_seq(0, tok)
    m.release_seq(1)                   # releasing a free slot is a no-op
    assert m.seq_lengths()[:2] == [40, -1]
    x = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, 2, dtype=torch.int32, device="cuda")
    with pytest.raises(b.DFError) as e:
        m.generate(x, -1, 0, out)
    assert e.value.status == b.DF_ERR_ARG
    with pytest.raises(b.DFError) as e:
        m.generate(x, 61, 0, torch.zeros(61, 2, dtype=torch.int32, device="cuda"))  # 40 + 61 > 100
    assert e.value.status == b.DF_ERR_CAPACITY
    assert m.seq_lengths()[:2] == [40, -1]
    with pytest.raises(b.DFError) as e:
        b.df_generate(m.ctx, x.data_ptr(), 2, 0, 0)   # no output buffer
    assert e.value.status == b.DF_ERR_ARG
    m.generate(x, 4, 0, out)
    m.sync()
    assert m.seq_lengths()[:2] == [44, -1]
    assert int(out[:, 0].min()) >= 0 and int(out[:, 0].max()) < cfg.vocab
    m.close()


@pytest.mark.parametrize("name", ["t_bf16_b1", "t_bf16_b9"])
def test_bounded_wait_that_runs_out_is_reported(name, cuda_device):
    """A bounded device wait that runs out is latched as DF_ERR_TIMEOUT and
    reported by df_sync, with the CUDA context left usable.  The wait is made
    to run out on purpose by the GEMM kernels' test hook
    (DF_TEST_GEMM_STALL_NS, read at df_create): every projection launch (the
    tensor-core GEMM, or the few-row GEMV at one sequence) first waits 1 ms on
    a barrier nothing arrives on, before it issues any copy, then stops; the
    tensor-core MMA issuer sees the abort flag and stops waiting too, so no
    copy or MMA is left in flight.  A fresh context created
    without the hook then decodes normally and matches the oracle."""
    import os
    import torch
    from dual_flow_transformer_decode_b300 import binding as b
    from oracle import Oracle
    cfg = dfsynth.get_config(name)
    w = Weights(cfg, 0)
    tok = dfsynth.tokens(cfg, 0)
    pre = torch.from_numpy(tok[:, :cfg.n_prefill].copy()).cuda()
    x = torch.from_numpy(tok[:, cfg.n_prefill].copy()).cuda()
    os.environ["DF_TEST_GEMM_STALL_NS"] = "1000000"
    try:
        m = _model(cfg)
    finally:
        del os.environ["DF_TEST_GEMM_STALL_NS"]
    m.prefill(pre)          # the batched prefill has its own GEMM kernel: unaffected
    m.sync()
    m.decode_step(x)
    with pytest.raises(b.DFError) as e:
        m.sync()
    assert e.value.status == b.DF_ERR_TIMEOUT
    # 104: the few-row GEMV (one sequence); 103: the tensor-core GEMM's
    # producer (9 sequences)
    assert f"detail {104 if cfg.batch == 1 else 103}" in str(e.value), str(e.value)
    m.sync()                # reported once: the latch is cleared, the context still answers
    m.close()
    m2 = _model(cfg)
    m2.prefill(pre)
    lp = torch.zeros(cfg.batch, cfg.vocab, device="cuda")
    m2.decode_step(x, lp)
    m2.sync()
    o = Oracle(cfg, w, cfg.batch)
    o.prefill(tok[:, :cfg.n_prefill])
    r = o.decode_step(tok[:, cfg.n_prefill])
    assert float(np.abs(lp.double().cpu().numpy() - r["logp_mix"]).max()) <= 2e-2
    m2.close()
