"""Oracle group advantage (float64). Test infrastructure only; see ``oracle/__init__.py``.

Sources, cited by page title and section:

* "03 Data Protocol and Batch Lifecycle" (verl source reading), *AgentLoop to trajectory
  value*: ``uid`` names one prompt group; ``rollout.n`` sessions per uid.
* same page, *response mask semantics*: GRPO's scalar advantage is broadcast to the tokens and
  multiplied by the response mask.
* "How a context-compaction step fits a variable number of rows into one batch",
  *Why the row count does not change the math*, item 2: the advantage is computed once per
  rollout and copied to all its rows; padding rows get 0.

The pages never print the formula. Reading (the standard group-normalised GRPO advantage):
``A_r = (R_r - mean_g) / (std_g + eps)`` over the rollouts of group g, with ``std`` the
unbiased (n-1) deviation by default. A group of one rollout, or one whose rewards are all
equal, has A = 0. Groups are consecutive runs of ``group_size`` rollouts.
"""
from __future__ import annotations

import math

import numpy as np


def group_advantage(rewards, group_size: int, eps: float, unbiased: bool = True) -> np.ndarray:
    """Per-rollout advantage; float64 arithmetic, float32 result (round to nearest even).

    Plain loops in the order a reader would write them: mean, then the squared deviations,
    then the scale. ``eps`` is used exactly as given (callers pass the float32 value the
    library receives).
    """
    rewards = [float(x) for x in rewards]
    n = len(rewards)
    if group_size <= 0 or n % group_size != 0:
        raise ValueError("rollouts must form whole groups")
    out = np.zeros(n, dtype=np.float32)
    eps = float(eps)
    for g0 in range(0, n, group_size):
        grp = rewards[g0:g0 + group_size]
        G = len(grp)
        if G < 2 and unbiased:
            continue  # unbiased std of a single sample is undefined: A = 0
        total = 0.0
        for x in grp:
            total = total + x
        mean = total / G
        ss = 0.0
        for x in grp:
            d = x - mean
            ss = ss + d * d
        var = ss / (G - 1) if unbiased else ss / G
        std = math.sqrt(var)
        for i, x in enumerate(grp):
            out[g0 + i] = np.float32((x - mean) / (std + eps))
    return out


def broadcast_to_tokens(adv_rollout, row_rollout, row_len) -> np.ndarray:
    """Copy each row's rollout advantage to all of that row's tokens (pad rows: -1 -> 0)."""
    parts = []
    for r, L in zip(row_rollout, row_len):
        a = np.float32(0.0) if r < 0 else np.float32(adv_rollout[r])
        parts.append(np.full(int(L), a, dtype=np.float32))
    return np.concatenate(parts) if parts else np.zeros(0, np.float32)
