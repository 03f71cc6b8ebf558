"""Shared test-side helpers for the GPU parity tests (test infrastructure; imports the oracle).

Tolerances (the loss and dlogits bars; ex2.approx is within 2^-22 relative, the exponent
argument (z - LSE) log2(e) carries <= |z - LSE| 2^-24 log2(e), the float32 LSE ~1e-6, bf16
rounding 2^-9):
* log-prob:   |d| <= 1e-5 * max(1, |ref|)
* token loss: |d| <= 1e-5 * |ref| + 1e-7 * |A|
* step loss:  |d| <= 1e-5 * max(|L_ref|, sum|m * l| / N)
* dlogits, every element, relative to its own value:
      bf16 output:  |d| <= 1e-2 * |ref| + 2^-120
      f32 output:   |d| <= 2e-5 * |ref| + 2^-120
  The 2^-120 floor only admits results that underflow: the kernels' ex2.approx.ftz returns 0
  below the smallest normal float (2^-126, which bf16 shares), so an element whose exact value
  is below 2^-126 |coef| may come back as 0; 2^-120 covers |coef| <= 64 and is far below any
  element that does not underflow.
  At the target element, where coef * (p_y - 1) cancels when p_y is near 1, a further
  1e-5 * |coef| (coef = m * A * r * g * scale: float32 rounding of p_y is relative to 1).
  With the entropy bonus, element v also carries ent * scale * p_v (z_v - E_p z), whose float32
  difference is exact only to ~2^-23 |z|: a further 1e-5 * p_v * sum_u |dz_u| (relative to the
  element's own probability, so a wrong small element still fails).
  The coefficient itself is a function of the float32 log-prob: c = A r g - kl_coef dk, with
  dc/dlogp = A r g (the ratio) + kl_coef e^(ref - logp) (KL k3; 0 for k1). A log-prob within its
  own bar (dlogp <= 1e-5 max(1, |logp|)) moves c by |dc/dlogp| dlogp, and every element of the
  row with it: a further (that / |c|) * |ref| per row (coef_err). It matters where c is small
  against its parts: a zero advantage with ref close to logp, or the KL term cancelling the
  surrogate.
Tokens whose float64 ratio lies within 1e-4 (relative) of a clip bound are ambiguous (float32
and float64 may take the clip decision differently); their dlogits row must equal the
oracle's row for one of the two decisions.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import advantage as OA
from oracle import loss as OL
from oracle import planner as OP

DLOGIT_REL = {"bf16": 1e-2, "f32": 2e-5}
UNDERFLOW_FLOOR = 2.0 ** -120
TARGET_COEF_TOL = 1e-5
ENTROPY_MASS_TOL = 1e-5


def oracle_logp(logits_host: np.ndarray, target: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Reference log-prob of every mask=1 token (float64), 0 elsewhere."""
    T = logits_host.shape[0]
    out = np.zeros(T)
    for t in range(T):
        if mask[t]:
            out[t] = OL.log_softmax_row(OL.as_f64(logits_host[t]))[int(target[t])]
    return out


class Case:
    """Inputs of one batch in input token order, on host (numpy) and device (torch)."""

    def __init__(self, wl, device="cuda", old_mode="noise", adv_override=None):
        self.wl = wl
        self.logits = W_make_logits(wl, device)
        self.logits_host = W_to_host(self.logits)
        self.target = wl.target
        self.mask = wl.mask
        self.adv_rollout = OA.group_advantage(wl.rewards, wl.group_size, np.float32(1e-6), True)
        self.adv_tok = OA.broadcast_to_tokens(self.adv_rollout, wl.row_rollout, wl.row_len)
        if adv_override is not None:
            self.adv_tok = adv_override.astype(np.float32)
        if old_mode == "none":
            self.old = None
        else:
            ref = oracle_logp(self.logits_host, wl.target, wl.mask)
            self.old = (ref + wl.old_noise.astype(np.float64)).astype(np.float32)
        dev = torch.device(device)
        self.d_target = torch.from_numpy(wl.target).to(dev)
        self.d_mask = torch.from_numpy(wl.mask).to(dev)
        self.d_adv = torch.from_numpy(self.adv_tok).to(dev)
        self.d_old = None if self.old is None else torch.from_numpy(self.old).to(dev)


def W_make_logits(wl, device):
    from rl_post_token_gb300 import workloads as W
    return W.make_logits(wl, device)


def W_to_host(t):
    from rl_post_token_gb300 import workloads as W
    return W.logits_to_host(t)


def oracle_run(case: Case, rows=None, scale_per_token=None, want_grad=True):
    """Oracle outputs for all tokens (or token subset `rows`) of a case."""
    idx = np.arange(case.logits_host.shape[0]) if rows is None else np.asarray(rows)
    s = np.ones(idx.shape[0]) if scale_per_token is None else scale_per_token[idx]
    T = idx.shape[0]
    V = case.wl.V
    out = {"loss_tok": np.zeros(T), "logp_tok": np.zeros(T), "ratio": np.ones(T),
           "clipped": np.zeros(T, bool), "coef": np.zeros(T), "target": case.target[idx]}
    if want_grad:
        out["dlogits"] = np.zeros((T, V))
    for k, t in enumerate(idx):
        old = None if case.old is None else float(case.old[t])
        z = OL.as_f64(case.logits_host[t]) if case.mask[t] else np.zeros(V)
        lt, lp, r, cl, dz = OL.token_objective(z, int(case.target[t]), old, float(case.adv_tok[t]),
                                               int(case.mask[t]), case.wl.eps, float(s[k]), want_grad)
        out["loss_tok"][k], out["logp_tok"][k], out["ratio"][k], out["clipped"][k] = lt, lp, r, cl
        if case.mask[t] and not cl:
            out["coef"][k] = float(case.adv_tok[t]) * r * float(s[k])
        if want_grad:
            out["dlogits"][k] = dz
    return out


def ambiguous_clip(ratio: np.ndarray, eps: float, rel=1e-4) -> np.ndarray:
    lo, hi = 1 - eps, 1 + eps
    return (np.abs(ratio - hi) <= rel * hi) | (np.abs(ratio - lo) <= rel * lo)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def row_probs(logits_host: np.ndarray) -> np.ndarray:
    """Softmax of every row (float64), from the oracle's log-softmax."""
    return np.stack([np.exp(OL.log_softmax_row(OL.as_f64(r))) for r in logits_host])


def dlogits_tol(ref, dtype, target=None, coef=None, probs=None, rel=None, coef_err=None):
    """Elementwise dlogits bar (see the module docstring): `rel` (default by output dtype)
    times each element's own magnitude, the underflow floor, the target-element term when
    `target` and `coef` are given, the entropy term when `probs` (row softmax) is given, and
    the coefficient's propagated error when `coef_err` (per row, absolute) and `coef` are."""
    r = DLOGIT_REL[dtype] if rel is None else rel
    tol = r * np.abs(ref) + UNDERFLOW_FLOOR
    if target is not None and coef is not None:
        rows = np.arange(ref.shape[0])
        tol[rows, target] += TARGET_COEF_TOL * np.abs(coef)
    if probs is not None:
        tol += ENTROPY_MASS_TOL * probs * np.sum(np.abs(ref), axis=1, keepdims=True)
    if coef_err is not None and coef is not None:
        c = np.abs(np.asarray(coef, dtype=np.float64))
        rel_row = np.where(c > 0, np.asarray(coef_err, dtype=np.float64) / np.where(c > 0, c, 1.0), 0.0)
        tol += rel_row[:, None] * np.abs(ref)
    return tol


def coef_logp_err(adv, ratio, clipped, mask, logp, scale, kl_kind=0, kl_coef=0.0, ref_logp=None):
    """Per token: |dc/dlogp| times the log-prob bar, times the grad scale (see the module
    docstring): the coefficient error a float32 log-prob within its own bar explains."""
    lp = np.asarray(logp, dtype=np.float64)
    d = (np.abs(np.asarray(adv, dtype=np.float64) * ratio) * (~np.asarray(clipped, bool))).astype(np.float64)
    if kl_kind == 2:
        d = d + kl_coef * np.exp(np.asarray(ref_logp, dtype=np.float64) - lp)
    return np.where(np.asarray(mask) != 0, d * 1e-5 * np.maximum(1.0, np.abs(lp)) * np.abs(scale), 0.0)


def _bad(got, ref, dtype, target, coef):
    return np.abs(got - ref) > dlogits_tol(ref, dtype, target, coef)


def assert_dlogits_close(got: np.ndarray, ref: np.ndarray, dtype: str, ok_rows=None, alt=None,
                         target=None, coef=None):
    """Elementwise dlogits bar; rows flagged in ok_rows may match `alt` instead of `ref`."""
    bad = _bad(got, ref, dtype, target, coef)
    if ok_rows is not None and alt is not None:
        bad2 = _bad(got, alt, dtype, target, coef)
        for t in np.nonzero(ok_rows)[0]:
            if not bad2[t].any():
                bad[t] = False
    if bad.any():
        t, v = np.argwhere(bad)[0]
        raise AssertionError(f"dlogits mismatch at ({t},{v}): got {got[t, v]!r} ref {ref[t, v]!r}; "
                             f"{int(bad.sum())} bad of {bad.size}")


def assert_tokens_close(got_loss, got_logp, ref, adv, mask):
    m = mask.astype(bool)
    dl = np.abs(got_logp - ref["logp_tok"])
    assert np.all(dl[m] <= 1e-5 * np.maximum(1.0, np.abs(ref["logp_tok"][m]))), float(dl[m].max())
    assert np.all(got_logp[~m] == 0)
    dloss = np.abs(got_loss - ref["loss_tok"])
    assert np.all(dloss <= 1e-5 * np.abs(ref["loss_tok"]) + 1e-7 * np.abs(adv)), float(dloss.max())
    assert np.all(got_loss[~m] == 0)


def plan_oracle(wl):
    return OP.plan(OP.PlanConfig(**wl.plan), wl.row_len, wl.row_valid, seg_counts=wl.seg_counts)
