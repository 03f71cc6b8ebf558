"""Host accumulation window in the library vs the oracle window: identical actions, scales,
counters and roll-up on seeded random chunk sequences with non-finite chunks. CPU only."""
import math

import numpy as np
import pytest

from oracle import window as OW


@pytest.mark.parametrize("seed", range(25))
def test_window_matches_oracle(grpo_lib, seed):
    from rl_post_token_gb300 import _lib
    rng = np.random.default_rng(seed)
    n_micro = int(rng.integers(1, 7))
    o, c = OW.Window(n_micro), _lib.Window(n_micro)
    for _ in range(int(rng.integers(10, 80))):
        finite = bool(rng.random() > 0.15)
        loss = float(rng.normal()) if finite else math.nan
        denom = int(rng.integers(0, 3000))
        ao, so = o.chunk(finite, loss, denom)
        ac, sc = c.grpo_window_chunk(finite, loss, denom)
        assert ao == ac and so == sc
    st = c.state
    assert (st["steps"], st["skipped_windows"], st["dropped_chunks"]) == (o.steps, o.skipped_windows, o.dropped_chunks)
    lo, do, so_ = o.rollup()
    lc, dc, sc_ = c.grpo_window_rollup()
    assert (do, so_) == (dc, sc_) and lc == pytest.approx(lo, rel=1e-15, abs=0)


def test_window_rejects_bad_arguments(grpo_lib):
    from rl_post_token_gb300 import _lib
    with pytest.raises(_lib.GrpoError):
        _lib.Window(0)
    w = _lib.Window(2)
    with pytest.raises(_lib.GrpoError):
        w.grpo_window_chunk(True, 1.0, -1)
