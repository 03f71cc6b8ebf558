"""The Python binding's own argument checks (it only marshals arguments, so these are the
layouts it refuses before calling the library). CPU tensors: no call reaches the device."""
import pytest
import torch

from rl_post_token_gb300 import _lib


def _side(T):
    return dict(target=torch.zeros(T, dtype=torch.int32), old_logp=None, adv_tok=torch.zeros(T),
                mask=torch.ones(T, dtype=torch.uint8), clip_eps=0.2, grad_scale=1.0, loss_tok=torch.zeros(T),
                logp_tok=None, acc=torch.zeros(_lib.ACC_BYTES, dtype=torch.uint8))


@pytest.mark.parametrize("bad", ["1d", "transposed", "dl_dtype", "dl_rows", "dl_transposed"])
def test_row_pass_binding_refuses_layouts(bad):
    lg = torch.zeros(4, 16, dtype=torch.bfloat16)
    dl = torch.zeros(4, 16, dtype=torch.bfloat16)
    if bad == "1d":
        lg = torch.zeros(64, dtype=torch.bfloat16)
    elif bad == "transposed":
        lg = torch.zeros(16, 4, dtype=torch.bfloat16).t()
    elif bad == "dl_dtype":
        dl = torch.zeros(4, 16, dtype=torch.float32)
    elif bad == "dl_rows":
        dl = torch.zeros(3, 16, dtype=torch.bfloat16)
    elif bad == "dl_transposed":
        dl = torch.zeros(16, 4, dtype=torch.bfloat16).t()
    with pytest.raises(ValueError, match="logits" if bad in ("1d", "transposed") else "dlogits"):
        _lib.grpo_logprob_loss_fwd_bwd(lg, dlogits=dl, **_side(4))


@pytest.mark.parametrize("bad, match", [("1d", "logits_host"), ("transposed", "logits_host"),
                                        ("staging_host", "staging")])
def test_host_entry_binding_refuses_layouts(bad, match):
    # (the staging-size and dlogits checks follow the staging buffer's, which needs a GPU)
    lg = torch.zeros(4, 16, dtype=torch.bfloat16)
    staging = torch.zeros(2 * 4 * 16 * 2, dtype=torch.uint8)  # a host buffer: refused
    if bad == "1d":
        lg = torch.zeros(64, dtype=torch.bfloat16)
    elif bad == "transposed":
        lg = torch.zeros(16, 4, dtype=torch.bfloat16).t()
    with pytest.raises(ValueError, match=match):
        _lib.grpo_logprob_loss_fwd_bwd_host(lg, dlogits=None, staging=staging, block_rows=4, **_side(4))


def test_status_error_carries_code_and_name():
    e = _lib.GrpoError(_lib.ERR_CAPACITY, "grpo_lmhead_loss_fwd_bwd")
    assert e.code == _lib.ERR_CAPACITY
    assert "grpo_lmhead_loss_fwd_bwd" in str(e)


def test_driver_refuses_short_accumulators_before_launching():
    # run_batch writes one 128-byte accumulator per optimizer step: a shorter buffer, or a
    # sequence-level mode without its weights, is refused before anything is enqueued
    from rl_post_token_gb300 import step as S
    from rl_post_token_gb300 import workloads as W
    wl = W.make_workload("tiny")
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid)
    assert bp.n_steps == 2
    kw = dict(logits=None, dlogits=None, target=None, old_logp=None, mask=None, adv_tok=None, loss_tok=None,
              logp_tok=None, clip_eps=0.2)
    with pytest.raises(ValueError, match="accs"):
        S.run_batch(bp, accs=torch.zeros(_lib.ACC_BYTES, dtype=torch.uint8), **kw)
    with pytest.raises(ValueError, match="w_tok"):
        S.run_batch(bp, accs=torch.zeros(2 * _lib.ACC_BYTES, dtype=torch.uint8),
                    agg=_lib.AGG_SEQ_MEAN_TOKEN_MEAN, **kw)
