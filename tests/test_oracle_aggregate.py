"""Pins of the oracle's loss aggregation modes (``oracle/aggregate.py``): a hand-worked step,
closed forms that relate the modes, linearity (the per-token scale is the derivative of the
step loss), the chain rule through the logits by central differences, and invariances."""
import numpy as np
import pytest

from oracle import aggregate as AG
from oracle import loss as OL

MODES = (AG.TOKEN_MEAN, AG.SEQ_MEAN_TOKEN_SUM, AG.SEQ_MEAN_TOKEN_MEAN)


def test_hand_worked_step():
    # row 0: three valid tokens with losses 1, 2, 3; row 1: one valid token (4) and one masked
    # token whose stored loss must be ignored; row 2: no valid token (not a sequence of the step)
    off = np.array([0, 3, 5, 7])
    mask = np.array([1, 1, 1, 1, 0, 0, 0], np.uint8)
    loss = np.array([1.0, 2.0, 3.0, 4.0, 99.0, 7.0, 7.0])
    assert AG.divisor(off, mask, AG.TOKEN_MEAN) == 4
    assert AG.divisor(off, mask, AG.SEQ_MEAN_TOKEN_SUM) == 2
    assert AG.aggregate(loss, off, mask, AG.TOKEN_MEAN) == 2.5              # 10 / 4
    assert AG.aggregate(loss, off, mask, AG.SEQ_MEAN_TOKEN_SUM) == 5.0      # (6 + 4) / 2
    assert AG.aggregate(loss, off, mask, AG.SEQ_MEAN_TOKEN_MEAN) == 3.0     # (6/3 + 4/1) / 2
    np.testing.assert_array_equal(AG.token_scale(off, mask, AG.SEQ_MEAN_TOKEN_MEAN),
                                  [1 / 6, 1 / 6, 1 / 6, 1 / 2, 1 / 2, 1 / 2, 1 / 2])


@pytest.mark.parametrize("L,R", [(1, 5), (7, 3), (16, 9)])
def test_equal_full_rows_closed_forms(L, R):
    rng = np.random.default_rng(L * 31 + R)
    off = np.arange(R + 1) * L
    mask = np.ones(R * L, np.uint8)
    loss = rng.normal(size=R * L)
    tm = AG.aggregate(loss, off, mask, AG.TOKEN_MEAN)
    assert AG.aggregate(loss, off, mask, AG.SEQ_MEAN_TOKEN_MEAN) == pytest.approx(tm, rel=1e-13, abs=1e-15)
    assert AG.aggregate(loss, off, mask, AG.SEQ_MEAN_TOKEN_SUM) == pytest.approx(L * tm, rel=1e-13, abs=1e-15)


def test_single_row():
    rng = np.random.default_rng(4)
    loss = rng.normal(size=11)
    mask = (rng.random(11) < 0.7).astype(np.uint8)
    mask[0] = 1
    off = np.array([0, 11])
    n = int(mask.sum())
    total = float(np.sum(loss[mask != 0]))
    assert AG.aggregate(loss, off, mask, AG.TOKEN_MEAN) == pytest.approx(total / n, rel=1e-14)
    assert AG.aggregate(loss, off, mask, AG.SEQ_MEAN_TOKEN_SUM) == pytest.approx(total, rel=1e-14)
    assert AG.aggregate(loss, off, mask, AG.SEQ_MEAN_TOKEN_MEAN) == pytest.approx(total / n, rel=1e-14)


@pytest.mark.parametrize("mode", MODES)
def test_token_scale_is_the_derivative(mode):
    # the step loss is linear in the per-token losses: bumping one valid token's loss by 1
    # moves it by exactly that token's scale; bumping a masked one moves nothing
    rng = np.random.default_rng(10 + mode)
    lens = rng.integers(1, 9, 6)
    off = np.concatenate([[0], np.cumsum(lens)])
    T = int(off[-1])
    mask = (rng.random(T) < 0.6).astype(np.uint8)
    mask[off[2]:off[3]] = 0   # one row with no valid token
    loss = rng.normal(size=T)
    base = AG.aggregate(loss, off, mask, mode)
    s = AG.token_scale(off, mask, mode)
    for t in range(T):
        bumped = loss.copy()
        bumped[t] += 1.0
        d = AG.aggregate(bumped, off, mask, mode) - base
        assert d == pytest.approx(s[t] if mask[t] else 0.0, abs=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_chain_rule_through_logits(mode):
    # d(step loss)/dz by central differences equals the objective's dlogits with the mode's
    # per-token scale
    rng = np.random.default_rng(20 + mode)
    lens = np.array([3, 1, 2])
    off = np.concatenate([[0], np.cumsum(lens)])
    T, V = int(off[-1]), 6
    z = rng.normal(size=(T, V))
    y = rng.integers(0, V, T)
    mask = np.array([1, 1, 0, 1, 1, 1], np.uint8)
    adv = rng.choice([-1.0, 0.7, 1.3], T)
    old = np.array([OL.log_softmax_row(z[t])[y[t]] for t in range(T)]) + rng.normal(0, 0.05, T)
    eps = 0.2
    s = AG.token_scale(off, mask, mode)
    out = OL.loss_fwd_bwd(z, y, old, adv, mask, eps, s, want_grad=True)

    def step_loss(zz):
        o = OL.loss_fwd_bwd(zz, y, old, adv, mask, eps, 1.0, want_grad=False)
        return AG.aggregate(o["loss_tok"], off, mask, mode)

    h = 1e-6
    for t in range(T):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[t, v] += h
            zm[t, v] -= h
            fd = (step_loss(zp) - step_loss(zm)) / (2 * h)
            assert fd == pytest.approx(out["dlogits"][t, v], abs=1e-7)


@pytest.mark.parametrize("mode", MODES)
def test_row_order_does_not_matter(mode):
    rng = np.random.default_rng(30 + mode)
    lens = rng.integers(1, 7, 5)
    off = np.concatenate([[0], np.cumsum(lens)])
    T = int(off[-1])
    mask = (rng.random(T) < 0.7).astype(np.uint8)
    loss = rng.normal(size=T)
    perm = rng.permutation(5)
    tok = np.concatenate([np.arange(off[r], off[r + 1]) for r in perm])
    off2 = np.concatenate([[0], np.cumsum(lens[perm])])
    a = AG.aggregate(loss, off, mask, mode)
    b = AG.aggregate(loss[tok], off2, mask[tok], mode)
    assert a == pytest.approx(b, rel=1e-14, abs=1e-15)


@pytest.mark.parametrize("mode", MODES)
def test_empty_step(mode):
    off = np.array([0, 2, 5])
    mask = np.zeros(5, np.uint8)
    loss = np.zeros(5)
    assert AG.divisor(off, mask, mode) == 0
    assert AG.aggregate(loss, off, mask, mode) == 0.0
    assert np.all(np.isfinite(AG.token_scale(off, mask, mode)))
