"""Seeded random cases of the row pass (grpo_logprob_loss_fwd_bwd and its _ex form) against the
float64 oracle.

Each case draws:
- a vocabulary size across the kernel shapes: the one-block kernels, the L2-resident kernel,
  and 2-, 3- and 4-CTA clusters;
- float32 or bf16 logits;
- logits and dlogits buffers whose rows are longer than V (the stride `ld`, `ld_out`);
- permuted execution order with padding rows (`tok_src`);
- masked tokens and a zero-advantage row;
- a regulariser: none, KL k3, the entropy bonus, or KL k1 with per-token weights.

The logits' columns past V hold NaN, so a read past the row fails the comparison. The dlogits'
columns past V hold a sentinel that must survive.

Tolerances are those of tests/_gpu_helpers.py: the per-element dlogits bar, the target term,
the entropy term, the coefficient's error propagated from the float32 log-prob, and tokens
whose ratio sits on a clip bound left out."""
import numpy as np
import pytest
import torch

from oracle import loss as OL
from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import workloads as W

from tests import _gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"
# vocabulary sizes: below and above the one-block and L2 limits, ragged and aligned cluster
# sizes, the product vocabulary, and one that needs four CTAs per row
V_CHOICES = [7, 300, 2053, 8200, 16384, 32776, 65544, 100003, 151936, 262144]


@pytest.fixture(scope="module", autouse=True)
def _built(grpo_lib):
    assert torch.cuda.is_available()
    return grpo_lib


def _draw(k):
    rng = np.random.default_rng(3000 + k)
    dtype = ("bf16", "f32")[k % 2]
    V = int(V_CHOICES[(k * 7 + int(rng.integers(0, 3))) % len(V_CHOICES)])
    rows = int(rng.choice([4, 8]))  # whole groups of 4 rollouts
    positions = int(rng.integers(3, 40)) if V < 200000 else int(rng.integers(3, 12))
    pad_in = int(rng.choice([0, 8, 3]))
    pad_out = int(rng.choice([0, 16, 5]))
    permuted = bool(rng.integers(0, 2))
    return rng, dtype, V, rows, positions, pad_in, pad_out, permuted


@pytest.mark.parametrize("k", range(16))
def test_rowpass_random_cases(k):
    rng, dtype, V, rows, positions, pad_in, pad_out, permuted = _draw(k)
    wl = W.make_workload("tiny", rows=rows, positions=positions, valid_lo=max(1, positions // 3), V=V,
                         dtype=dtype, seed=4000 + k, std=2.5)
    case = H.Case(wl)
    T = wl.T
    adv = case.adv_tok.copy()
    adv[:positions] = 0.0  # the first row: a group whose rewards were all equal
    kind = k % 4
    kl = (0, _lib.KL_K3, 0, _lib.KL_K1)[kind]
    ent = 0.02 if kind == 2 else 0.0
    ref_lp = (case.old + rng.normal(0, 0.3, T)).astype(np.float32)
    w_tok = rng.choice([1.0, 0.5, 0.2], T).astype(np.float32) if kind == 3 else None
    gs = np.float32(1.0 / max(int(wl.mask.sum()), 1))

    # execution order: a permutation of the tokens plus two padding rows, or the input order
    if permuted:
        perm = rng.permutation(T)
        pads = rng.choice(T, 2)
        src = np.concatenate([perm, pads])
        tok_src = np.concatenate([perm, -1 - pads]).astype(np.int64)
    else:
        src = np.arange(T)
        tok_src = None
    Te = len(src)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    big_in = torch.full((Te, V + pad_in), float("nan"), dtype=tdt, device=DEV)
    big_in[:, :V] = case.logits[torch.from_numpy(src).to(DEV)]
    big_out = torch.full((Te, V + pad_out), 7.0, dtype=tdt, device=DEV)
    lg, dl = big_in[:, :V], big_out[:, :V]
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    ent_t = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    terms = None
    if kind:
        terms = dict(kl_kind=kl, kl_coef=0.1, ref_logp=t(ref_lp) if kl else None, ent_coef=ent,
                     entropy_tok=ent_t if kind == 2 else None, w_tok=t(w_tok))
    _lib.grpo_logprob_loss_fwd_bwd(lg, case.d_target, case.d_old, t(adv), case.d_mask, wl.eps, float(gs), dl, loss,
                                   logp, acc, tok_src=t(tok_src), terms=terms)
    torch.cuda.synchronize()

    scale = (gs * w_tok).astype(np.float64) if w_tok is not None else float(gs)
    oterms = None if not kind else dict(kl_kind=kl, kl_coef=float(np.float32(0.1)), ref=ref_lp.astype(np.float64),
                                        ent_coef=float(np.float32(ent)))
    ref = OL.loss_fwd_bwd(case.logits_host, wl.target, case.old, adv, wl.mask, wl.eps, scale, True, oterms)
    m = wl.mask.astype(bool)
    gl, gp = H.to_f64(loss), H.to_f64(logp)
    assert np.all(np.abs(gp[m] - ref["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref["logp_tok"][m])))
    assert np.all(gp[~m] == 0) and np.all(gl[~m] == 0)
    assert np.all(np.abs(gl - ref["loss_tok"]) <= 1e-5 * np.abs(ref["loss_tok"]) + 1e-6)
    if kind == 2:
        ge = H.to_f64(ent_t)
        assert np.all(np.abs(ge[m] - ref["entropy"][m]) <= 1e-5 * np.maximum(1, ref["entropy"][m]))
    # dlogits in execution order: a token's row, or zeros for a padding row
    got = H.to_f64(dl)
    live = src[:T] if permuted else src
    want = ref["dlogits"][live]
    # each token's gradient coefficient (the target element's cancellation bar): the surrogate's
    # A r g, less the KL term's kl_coef * dk/dlogp, times the token's grad scale
    c = np.where(m & ~ref["clipped"], adv * ref["ratio"], 0.0)
    if kl == _lib.KL_K3:
        c = c - np.where(m, float(np.float32(0.1)) * (1.0 - np.exp(ref_lp - ref["logp_tok"])), 0.0)
    elif kl == _lib.KL_K1:
        c = c - np.where(m, float(np.float32(0.1)), 0.0)
    coef = (c * scale)[live]
    probs = H.row_probs(case.logits_host[live]) if kind == 2 else None
    cerr = H.coef_logp_err(adv, ref["ratio"], ref["clipped"], wl.mask, ref["logp_tok"], scale, kl,
                           float(np.float32(0.1)), ref_lp)[live]
    tol = H.dlogits_tol(want, dtype, target=wl.target[live], coef=coef, probs=probs, coef_err=cerr)
    bad = np.abs(got[:T] - want) > tol
    bad[H.ambiguous_clip(ref["ratio"][live], wl.eps)] = False
    if bad.any():
        r = np.unique(np.argwhere(bad)[:, 0])[:4]
        tok = live[r]
        detail = [dict(row=int(i), tok=int(j), adv=float(adv[j]), mask=int(wl.mask[j]), ratio=float(ref["ratio"][j]),
                       clipped=bool(ref["clipped"][j]), coef=float(coef[i]), got_sum=float(np.abs(got[i]).sum()),
                       want_sum=float(np.abs(want[i]).sum()), got0=float(got[i, 0]), want0=float(want[i, 0]))
                  for i, j in zip(r, tok)]
        raise AssertionError((k, int(bad.sum()), detail))
    if permuted:
        assert np.all(got[T:] == 0)
    # nothing written past V in any dlogits row
    if pad_out:
        assert torch.all(big_out[:, V:] == 7.0)
    res = _lib.grpo_finish_step(acc, loss)
    assert res["status"] == 0 and res["n_valid"] == int(wl.mask.sum()) and res["kernel_flags"] == 0
    assert res["n_tokens"] == Te
