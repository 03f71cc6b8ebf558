"""Pins for the oracle accumulation window against the pages' descriptions. CPU only."""
import math

import pytest

from oracle import window as OW


def test_poisoned_window_drops_the_rest_of_its_chunks():
    # four chunks per window; the third chunk of the first window is non-finite: the window is
    # discarded and its fourth chunk dropped; the next window trains normally and steps
    w = OW.Window(4)
    seq = [(True, 1.0, 10), (True, 1.0, 10), (False, math.nan, 10), (True, 1.0, 10),
           (True, 2.0, 5), (True, 2.0, 5), (True, 2.0, 5), (True, 2.0, 5)]
    acts = [w.chunk(*c)[0] for c in seq]
    assert acts == [OW.ACCUMULATE, OW.ACCUMULATE, OW.DISCARD, OW.DROP,
                    OW.ACCUMULATE, OW.ACCUMULATE, OW.ACCUMULATE, OW.STEP]
    # the abandoned window's divisor did not leak into the next one
    w2 = OW.Window(4)
    scales = [w2.chunk(*c)[1] for c in seq]
    assert scales[-1] == pytest.approx(1 / 20)
    assert (w.steps, w.skipped_windows, w.dropped_chunks) == (1, 1, 1)


def test_single_chunk_windows_lose_nothing_after_a_skip():
    w = OW.Window(1)
    acts = [w.chunk(True, 1.0, 3)[0], w.chunk(False, math.nan, 3)[0], w.chunk(True, 1.0, 3)[0]]
    assert acts == [OW.STEP, OW.DISCARD, OW.STEP]
    assert w.dropped_chunks == 0


def test_last_chunk_poisoned_drops_nothing_more():
    w = OW.Window(2)
    acts = [w.chunk(True, 1.0, 1)[0], w.chunk(False, 0.0, 1)[0], w.chunk(True, 1.0, 1)[0],
            w.chunk(True, 1.0, 1)[0]]
    assert acts == [OW.ACCUMULATE, OW.DISCARD, OW.ACCUMULATE, OW.STEP]


def test_step_scale_is_one_over_guarded_sum():
    w = OW.Window(2)
    w.chunk(True, 0.0, 0)
    act, scale = w.chunk(True, 0.0, 0)
    assert act == OW.STEP and scale == 1.0  # max(sum, 1): an all-empty window scales by 1


def test_rollup_is_token_weighted_not_mean_of_means():
    # unequal chunks: (loss 1 over 10 tokens, loss 3 over 30) -> 100 / 40 = 2.5, not 2.0
    w = OW.Window(2)
    w.chunk(True, 1.0, 10)
    w.chunk(True, 3.0, 30)
    loss, denom, steps = w.rollup()
    assert loss == pytest.approx(2.5) and denom == 40 and steps == 1
    # equal chunks cannot tell the two apart (which is why an acceptance run caught it)
    w = OW.Window(2)
    w.chunk(True, 1.0, 10)
    w.chunk(True, 3.0, 10)
    assert w.rollup()[0] == pytest.approx(2.0)
