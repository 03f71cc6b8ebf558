"""GPU parity of the loss aggregation modes through the C ABI and the driver loop: the per-token
gradient scales (grad_scale times the planner's per-token weights), the dlogits and the step
losses under seq-mean-token-sum and seq-mean-token-mean, against the oracle's definitions
(``oracle/aggregate.py``) applied step by step; plus chunk invariance and the deferred mode."""
import numpy as np
import pytest
import torch

from oracle import aggregate as AG
from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import step as S
from rl_post_token_gb300 import workloads as W

from tests import _gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built(grpo_lib):
    assert torch.cuda.is_available()
    return grpo_lib


def _workload(kind, agg):
    if kind == "fixed":
        # equal row lengths, random valid prefixes (some rows with none): the modes differ
        return W.make_workload("tiny", rows=8, positions=24, valid_lo=0, V=32776, dtype="bf16", seed=70 + agg,
                               std=2.0, mini=4, micro=2)
    # token-budget bins: exec order differs from input order, weights read through the index
    return W.make_workload("dynamic", rows=16, len_hi=64, median=20, max_token_len=160, V=4104, seed=80 + agg)


def _run(case, wl, agg, micro=None, deferred=False):
    plan = dict(wl.plan) if micro is None else dict(wl.plan, micro=micro)
    bp = S.plan_batch(plan, wl.row_len, wl.row_valid, wl.seg_counts)
    div, w = bp.token_weights(agg)
    w_d = torch.from_numpy(w).to(DEV) if agg == _lib.AGG_SEQ_MEAN_TOKEN_MEAN else None
    Te = bp.exec_tokens
    src = np.arange(Te) if bp.tok_src is None else bp.tok_src
    logits = case.logits[torch.from_numpy(np.where(src >= 0, src, -1 - src)).to(DEV)]
    dl = torch.empty_like(logits)
    loss = torch.full((wl.T,), -7.0, device=DEV)
    logp = torch.full((wl.T,), -7.0, device=DEV)
    accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
    S.run_batch(bp, logits=logits, dlogits=dl, target=case.d_target, old_logp=case.d_old, mask=case.d_mask,
                adv_tok=case.d_adv, loss_tok=loss, logp_tok=logp, accs=accs, clip_eps=wl.eps,
                tok_src=None if bp.tok_src is None else torch.from_numpy(bp.tok_src).to(DEV),
                deferred=deferred, agg=agg, w_tok=w_d)
    torch.cuda.synchronize()
    return bp, div, src, dl, loss, logp, S.read_results(accs, bp.n_steps)


def _oracle_scales(bp, wl, agg):
    """Per-token dL/dl_t of every optimizer step, by the oracle's definition, input order."""
    s = np.zeros(wl.T)
    div = []
    for k in range(bp.n_steps):
        r0, r1 = bp.plan["step_in_row_off"][k], bp.plan["step_in_row_off"][k + 1]
        off = bp.row_tok_off[r0:r1 + 1] - bp.row_tok_off[r0]
        t0, t1 = bp.step_tok_range[k]
        s[t0:t1] = AG.token_scale(off, wl.mask[t0:t1], agg)
        div.append(AG.divisor(off, wl.mask[t0:t1], agg))
    return s, div


@pytest.mark.parametrize("kind", ["fixed", "dynamic"])
@pytest.mark.parametrize("agg", [_lib.AGG_SEQ_MEAN_TOKEN_SUM, _lib.AGG_SEQ_MEAN_TOKEN_MEAN])
def test_seq_aggregation_matches_oracle(kind, agg):
    wl = _workload(kind, agg)
    case = H.Case(wl)
    bp, div, src, dl, loss, logp, res = _run(case, wl, agg)
    scales, odiv = _oracle_scales(bp, wl, agg)
    assert list(div) == odiv
    ref = H.oracle_run(case, scale_per_token=scales)
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, case.adv_tok, case.mask)
    # dlogits, exec rows mapped back to input order (padding rows: none in these plans)
    got = np.zeros_like(ref["dlogits"])
    got[src] = H.to_f64(dl)
    H.assert_dlogits_close(got, ref["dlogits"], "bf16", target=ref["target"],
                           coef=np.abs(case.adv_tok * ref["ratio"] * scales) * case.mask)
    for k in range(bp.n_steps):
        r0, r1 = bp.plan["step_in_row_off"][k], bp.plan["step_in_row_off"][k + 1]
        off = bp.row_tok_off[r0:r1 + 1] - bp.row_tok_off[r0]
        t0, t1 = bp.step_tok_range[k]
        want = AG.aggregate(ref["loss_tok"][t0:t1], off, wl.mask[t0:t1], agg)
        scale_abs = np.sum(np.abs(ref["loss_tok"][t0:t1]) * scales[t0:t1])
        assert res[k]["status"] == 0 and res[k]["n_valid"] == int(wl.mask[t0:t1].sum())
        assert abs(res[k]["loss"] - want) <= 1e-5 * max(abs(want), scale_abs) + 1e-12


def test_token_mean_through_the_weighted_path_equals_plain():
    # TOKEN_MEAN through the weighted entry points (weights all 1, divisor N) matches the plain
    # path: the weighted kernel instance sums a row in 16-element blocks instead of 32, so the
    # LSE may differ in its last bit; counts are identical, losses agree within the per-token
    # parity bar and dlogits to one bf16 rounding step
    wl = _workload("fixed", 0)
    case = H.Case(wl)
    outs = []
    for w in (None, "ones"):
        bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid)
        dl = torch.empty_like(case.logits)
        loss = torch.empty(wl.T, device=DEV)
        accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
        w_d = None if w is None else torch.ones(wl.T, device=DEV)
        S.run_batch(bp, logits=case.logits, dlogits=dl, target=case.d_target, old_logp=case.d_old,
                    mask=case.d_mask, adv_tok=case.d_adv, loss_tok=loss, logp_tok=None, accs=accs,
                    clip_eps=wl.eps, agg=_lib.AGG_TOKEN_MEAN, w_tok=w_d)
        torch.cuda.synchronize()
        outs.append((dl.float().clone(), loss.clone(), S.read_results(accs, bp.n_steps)))
    (d0, l0, r0), (d1, l1, r1) = outs
    # one bf16 step (2^-7 relative at most) on every element, plus a little at the target
    # element only, where coef * (p_y - 1) cancels
    tol = 2.0 ** -7 * d0.abs() + H.UNDERFLOW_FLOOR
    rows = torch.arange(wl.T, device=d0.device)
    tgt = case.d_target.long()
    tol[rows, tgt] += H.TARGET_COEF_TOL * d0.abs().amax(dim=1)
    assert torch.all((d1 - d0).abs() <= tol)
    # a last-bit LSE difference moves log p by ~1e-6 and the loss by as much relative: the
    # per-token parity bar
    assert torch.all((l1 - l0).abs() <= 1e-5 * l0.abs() + 1e-7)
    for a, b in zip(r0, r1):
        for k in ("n_valid", "n_clipped", "n_nonfinite", "n_tokens", "status", "kernel_flags"):
            assert a[k] == b[k], k
        assert abs(a["loss"] - b["loss"]) <= 1e-5 * max(abs(a["loss"]), 1e-6)


@pytest.mark.parametrize("agg", [_lib.AGG_SEQ_MEAN_TOKEN_SUM, _lib.AGG_SEQ_MEAN_TOKEN_MEAN])
def test_seq_aggregation_chunked_equals_unchunked_bitwise(agg):
    wl = _workload("fixed", agg)
    case = H.Case(wl)
    a = _run(case, wl, agg, micro=1)
    b = _run(case, wl, agg, micro=4)
    assert torch.equal(a[3].view(torch.int16), b[3].view(torch.int16))
    assert torch.equal(a[4], b[4])
    assert a[6] == b[6]


def test_seq_mean_token_mean_deferred_matches_direct():
    agg = _lib.AGG_SEQ_MEAN_TOKEN_MEAN
    wl = _workload("fixed", agg)
    case = H.Case(wl)
    _, _, _, dl_d, _, _, res_d = _run(case, wl, agg, deferred=True)
    bp, _, _, dl, _, _, res = _run(case, wl, agg)
    for k in range(bp.n_steps):
        assert res_d[k]["status"] == 0
        assert res_d[k]["loss"] == res[k]["loss"]
    # two bf16 roundings in the deferred path (before and after the 1/B scale)
    got, want = H.to_f64(dl_d), H.to_f64(dl)
    tol = H.dlogits_tol(want, "bf16", rel=2e-2)
    tol[np.arange(wl.T), wl.target] += H.TARGET_COEF_TOL * np.max(np.abs(want), axis=1)
    assert np.all(np.abs(got - want) <= tol)
