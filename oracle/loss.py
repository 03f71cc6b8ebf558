"""Oracle policy loss and its gradient w.r.t. the logits (float64).

Test infrastructure only; see ``oracle/__init__.py``.

Sources, cited by page title and section:

* "Sizing mini-batches and micro-batches" (cosmos posttrain batching how-to):
  - *The problem*: the cost is the log-softmax over the vocabulary for every completion token.
  - *The hard part: deferred normalization*: the loss is a token mean -- the per-token loss
    summed over the whole optimizer step, divided once by N, the number of valid (masked-in)
    completion positions; ``max(N, 1)`` guards an all-empty step; gradients are linear, so
    the chunk sums over N equal the gradient of the un-chunked step.
  - *pi_old must be frozen across the window*: the ratio is taken against pi_old, the clip
    uses an epsilon, with pi_old = the current policy the ratio is exp(0) = 1.
  - *Metric roll-up*: counts are summed; the loss is token-weighted.
* "03 Data Protocol and Batch Lifecycle" (verl source reading), *response mask semantics*:
  the policy loss accumulates only over response_mask = 1 tokens, and the advantage is
  broadcast to tokens and multiplied by the mask.
* "22-mini-batch-micro-batch-dynamic-batch-size的区别" (verl batching article), section 5:
  token-mean normalisation by the step's global token count.

The pages never print the surrogate. Reading (standard PPO clip, symmetric epsilon), for a
token with logits z, target y, pi_old log-prob ``old``, advantage A and mask m:

    LSE  = max(z) + log(sum(exp(z - max(z))))
    logp = z[y] - LSE
    r    = exp(logp - old)                       (r = 1 when there is no pi_old)
    l    = -min(r*A, clip(r, 1-eps, 1+eps)*A)
    loss_t = m * l
    g    = 0 if (A > 0 and r > 1+eps) or (A < 0 and r < 1-eps) else 1
    dloss_t/dz = m * A * r * g * (softmax(z) - onehot(y))

and the step loss is sum(loss_t) / max(N, 1), with dlogits scaled by the same 1/max(N, 1)
(``scale``). Masked tokens are not policy actions: their loss, log-prob output and dlogits
are 0 and their logits are never read.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def as_f64(logits: np.ndarray) -> np.ndarray:
    """Logits given as float32/float64 values or as bfloat16 bit patterns (uint16)."""
    if logits.dtype == np.uint16:
        return bf16_bits_to_f64(logits)
    return logits.astype(np.float64)


def log_softmax_row(z: np.ndarray) -> np.ndarray:
    # (z - max) - log sum exp(z - max): the definition z - log sum exp(z), written so that no
    # large quantity is subtracted from another (exact under any shift that keeps z exact)
    m = np.max(z)
    d = z - m
    return d - math.log(float(np.sum(np.exp(d))))


KL_NONE, KL_K1, KL_K3 = 0, 1, 2


def token_objective(z, y, old, adv, mask, eps, scale=1.0, want_grad=True, terms=None):
    """One token row. Returns (loss_t, logp, r, clipped, dz or None).

    ``terms`` (optional dict) adds the regularisers that the verl batching article (section 5)
    sends through the same token-mean aggregation; the pages give no formula, so the reading is
    the usual one:
      kl_coef * k(logp, ref)  with k1 = logp - ref, or k3 = exp(ref - logp) - (ref - logp) - 1
                              (kl_kind 1 or 2, ``ref`` the reference policy's log-prob);
      - ent_coef * H          with H = -sum_v p_v log p_v (an entropy bonus).
    Their gradients w.r.t. the logits: dk/dz = (dk/dlogp) (onehot - p) and
    dH/dz_v = -p_v (z_v - sum_u p_u z_u). The entropy is returned as terms["entropy"].
    """
    V = z.shape[0]
    if not mask:
        if terms is not None:
            terms["entropy"] = 0.0
        return 0.0, 0.0, 1.0, False, (np.zeros(V) if want_grad else None)
    z = np.asarray(z, dtype=np.float64)
    lsm = log_softmax_row(z)
    logp = float(lsm[y])
    r = 1.0 if old is None else math.exp(logp - float(old))
    A = float(adv)
    eps = float(eps)
    lo, hi = 1.0 - eps, 1.0 + eps
    rc = min(max(r, lo), hi)
    loss_t = -min(r * A, rc * A)
    clipped = (A > 0 and r > hi) or (A < 0 and r < lo)
    g = 0.0 if clipped else 1.0
    c = A * r * g          # d(loss)/dz = c * (p - onehot) for the surrogate
    ent_coef = 0.0
    if terms is not None:
        kind = int(terms.get("kl_kind", KL_NONE))
        if kind != KL_NONE:
            d = float(terms["ref"]) - logp
            if kind == KL_K1:
                k, dk = -d, 1.0
            else:
                k, dk = math.exp(d) - d - 1.0, 1.0 - math.exp(d)
            beta = float(terms.get("kl_coef", 0.0))
            loss_t += beta * k
            c -= beta * dk
        ent_coef = float(terms.get("ent_coef", 0.0))
        p = np.exp(lsm)
        # p log p -> 0 as p -> 0: elements without mass (-inf logits) add nothing
        with np.errstate(invalid="ignore"):
            H = -float(np.sum(np.where(p > 0, p * lsm, 0.0)))
        terms["entropy"] = H
        loss_t -= ent_coef * H
    dz = None
    if want_grad:
        p = np.exp(lsm)
        dz = float(scale) * c * p
        dz[y] -= float(scale) * c
        if ent_coef != 0.0:
            with np.errstate(invalid="ignore"):
                ez = float(np.sum(np.where(p > 0, p * z, 0.0)))
                dz += float(scale) * ent_coef * np.where(p > 0, p * (z - ez), 0.0)
    return loss_t, logp, r, clipped, dz


def loss_fwd_bwd(logits, target, old_logp, adv_tok, mask, eps, scale=1.0, want_grad=True, terms=None):
    """All token rows of ``logits`` ([T, V], float or bf16 bits).

    Returns dict with float64 ``loss_tok``, ``logp_tok``, ``ratio``, bool ``clipped`` and,
    if ``want_grad``, float64 ``dlogits`` [T, V]. ``scale`` is one gradient scale for every
    token or an array of per-token scales (an aggregation mode's dL/dl_t). ``terms`` =
    dict(kl_kind, kl_coef, ref (array per token), ent_coef) adds the regularisers of
    ``token_objective`` (output ``entropy``).
    """
    T = logits.shape[0]
    V = logits.shape[1] if logits.ndim == 2 else 0
    out = {
        "loss_tok": np.zeros(T), "logp_tok": np.zeros(T), "ratio": np.ones(T),
        "clipped": np.zeros(T, dtype=bool),
    }
    if want_grad:
        out["dlogits"] = np.zeros((T, V))
    if terms is not None:
        out["entropy"] = np.zeros(T)
    for t in range(T):
        old = None if old_logp is None else old_logp[t]
        z = as_f64(logits[t]) if mask[t] else np.zeros(V)
        tt = None
        if terms is not None:
            tt = dict(kl_kind=terms.get("kl_kind", 0), kl_coef=terms.get("kl_coef", 0.0),
                      ent_coef=terms.get("ent_coef", 0.0),
                      ref=None if terms.get("ref") is None else terms["ref"][t])
        st = scale[t] if np.ndim(scale) else scale
        lt, lp, r, cl, dz = token_objective(z, int(target[t]), old, adv_tok[t], int(mask[t]),
                                            eps, st, want_grad, tt)
        if tt is not None:
            out["entropy"][t] = tt["entropy"]
        out["loss_tok"][t] = lt
        out["logp_tok"][t] = lp
        out["ratio"][t] = r
        out["clipped"][t] = cl
        if want_grad:
            out["dlogits"][t] = dz
    return out


def finish_step(loss_tok, mask, clipped=None):
    """Step metrics: loss = sum(loss_t) / max(N, 1), N = sum(mask); counts are sums."""
    mask = np.asarray(mask)
    n_valid = int(np.sum(mask != 0))
    loss_sum = math.fsum(float(x) for x in np.asarray(loss_tok, dtype=np.float64))
    res = {"loss_sum": loss_sum, "loss": loss_sum / max(n_valid, 1), "n_valid": n_valid}
    if clipped is not None:
        n_clip = int(np.sum(np.asarray(clipped) & (mask != 0)))
        res["n_clipped"] = n_clip
        res["clipfrac"] = n_clip / max(n_valid, 1)
    return res


def lmhead_fwd_bwd(h, W, target, old_logp, adv_tok, mask, eps, scale=1.0, rows=None, want_dw=True, terms=None):
    """Fused LM-head variant: the same objective with the logits produced by z = h W^T.

    ``h`` [T, H] and ``W`` [V, H] are bfloat16 bit patterns (uint16) or floats. Computes, in
    float64, z = h W^T, then the token objective above, then the two backward products
    d_h = dz W and dW = dz^T h. ``rows`` restricts the work to a subset of tokens (d_h rows
    and per-token outputs only; dW needs every token and is then skipped). ``scale`` and
    ``terms`` are those of ``loss_fwd_bwd`` (a per-token scale array, the regularisers; the
    reference log-probs ``terms["ref"]`` indexed like the tokens).
    """
    hf = as_f64(h)
    Wf = as_f64(W)
    T = hf.shape[0]
    idx = np.arange(T) if rows is None else np.asarray(rows)
    z = hf[idx] @ Wf.T
    sc = np.asarray(scale)[idx] if np.ndim(scale) else scale
    tt = None
    if terms is not None:
        tt = dict(terms)
        if tt.get("ref") is not None:
            tt["ref"] = np.asarray(tt["ref"])[idx]
    out = loss_fwd_bwd(z, np.asarray(target)[idx], None if old_logp is None else np.asarray(old_logp)[idx],
                       np.asarray(adv_tok)[idx], np.asarray(mask)[idx], eps, sc, want_grad=True, terms=tt)
    dz = out.pop("dlogits")
    out["d_h"] = dz @ Wf
    if want_dw and rows is None:
        out["dW"] = dz.T @ hf
    return out
