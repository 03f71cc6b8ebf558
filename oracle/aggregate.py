"""Oracle of the loss aggregation modes: how one optimizer step's per-token losses become the
step loss, and the per-token gradient scale each mode implies. Test infrastructure only; see
``oracle/__init__.py``.

Sources, cited by page title and section:

* "Sizing mini-batches and micro-batches", *The hard part: deferred normalization*: the GRPO
  loss is a token mean over the whole step, divided once by N (valid completion positions),
  guarded by max(N, 1).
* "22-mini-batch-micro-batch-dynamic-batch-size的区别" (verl batching article), section 5:
  the aggregation function divides token-mean by the global token count and the
  sequence-level modes by the global batch size (the number of sequences); a data-parallel
  factor compensates for mean-reduced gradients across ranks (1 on one GPU).

The pages name the sequence-level modes without printing them. Reading (the two usual ones),
for the rows (sequences) of one step, n_r = valid tokens of row r, N = sum n_r, and
B = rows with n_r >= 1 (a row with no valid token -- a padding row or an empty completion --
is not a sequence of the step):

    TOKEN_MEAN          (0)  L = sum_r sum_{t in r} l_t / max(N, 1)
    SEQ_MEAN_TOKEN_SUM  (1)  L = sum_r (sum_{t in r} l_t) / max(B, 1)
    SEQ_MEAN_TOKEN_MEAN (2)  L = sum_r (sum_{t in r} l_t / max(n_r, 1)) / max(B, 1)

(l_t = m_t * loss_t, zero on masked tokens). Each is linear in the l_t, so dL/dl_t is the
per-token scale s_t: 1/max(N,1), 1/max(B,1) and 1/(max(n_r,1) max(B,1)) respectively.
"""
from __future__ import annotations

import math

import numpy as np

TOKEN_MEAN, SEQ_MEAN_TOKEN_SUM, SEQ_MEAN_TOKEN_MEAN = 0, 1, 2


def _rows(row_tok_off, mask):
    off = np.asarray(row_tok_off, dtype=np.int64)
    m = np.asarray(mask)
    n_r = np.array([int(np.sum(m[off[r]:off[r + 1]] != 0)) for r in range(off.shape[0] - 1)], dtype=np.int64)
    return off, m, n_r


def divisor(row_tok_off, mask, mode):
    """The step's divisor: N for TOKEN_MEAN, B for the sequence-level modes."""
    _, _, n_r = _rows(row_tok_off, mask)
    if mode == TOKEN_MEAN:
        return int(n_r.sum())
    if mode in (SEQ_MEAN_TOKEN_SUM, SEQ_MEAN_TOKEN_MEAN):
        return int(np.sum(n_r >= 1))
    raise ValueError("unknown aggregation mode")


def aggregate(loss_tok, row_tok_off, mask, mode):
    """The step loss of ``mode`` from per-token losses in input order, summed row by row."""
    off, m, n_r = _rows(row_tok_off, mask)
    lt = np.asarray(loss_tok, dtype=np.float64)
    row_sums = [math.fsum(float(lt[t]) for t in range(off[r], off[r + 1]) if m[t] != 0)
                for r in range(n_r.shape[0])]
    if mode == TOKEN_MEAN:
        return math.fsum(row_sums) / max(int(n_r.sum()), 1)
    B = int(np.sum(n_r >= 1))
    if mode == SEQ_MEAN_TOKEN_SUM:
        return math.fsum(row_sums) / max(B, 1)
    if mode == SEQ_MEAN_TOKEN_MEAN:
        return math.fsum(row_sums[r] / max(int(n_r[r]), 1) for r in range(n_r.shape[0])) / max(B, 1)
    raise ValueError("unknown aggregation mode")


def token_scale(row_tok_off, mask, mode):
    """dL/dl_t for every token of the step (float64, input order)."""
    off, m, n_r = _rows(row_tok_off, mask)
    T = int(off[-1])
    s = np.zeros(T)
    B = max(int(np.sum(n_r >= 1)), 1)
    for r in range(n_r.shape[0]):
        if mode == TOKEN_MEAN:
            v = 1.0 / max(int(n_r.sum()), 1)
        elif mode == SEQ_MEAN_TOKEN_SUM:
            v = 1.0 / B
        elif mode == SEQ_MEAN_TOKEN_MEAN:
            v = 1.0 / (max(int(n_r[r]), 1) * B)
        else:
            raise ValueError("unknown aggregation mode")
        s[off[r]:off[r + 1]] = v
    return s
