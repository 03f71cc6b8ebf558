"""Pins for the oracle group advantage: hand-worked values and numpy's mean/std. CPU only."""
import numpy as np
import pytest

from oracle.advantage import broadcast_to_tokens, group_advantage

EPS = np.float32(1e-6)


def test_hand_case_unbiased():
    # rewards [1,0,0,0]: mean 0.25; squared deviations 0.5625 + 3 * 0.0625 = 0.75;
    # unbiased variance 0.75 / 3 = 0.25, std 0.5; A = (R - 0.25) / (0.5 + eps)
    a = group_advantage([1, 0, 0, 0], 4, EPS, unbiased=True)
    e = float(EPS)
    want = np.array([0.75 / (0.5 + e), -0.25 / (0.5 + e), -0.25 / (0.5 + e), -0.25 / (0.5 + e)], np.float32)
    assert np.array_equal(a, want)
    assert abs(a[0] - 1.5) < 1e-5 and abs(a[1] + 0.5) < 1e-5


def test_hand_case_biased():
    # biased variance 0.75 / 4 = 0.1875, std = sqrt(3)/4
    a = group_advantage([1, 0, 0, 0], 4, 0.0, unbiased=False)
    s = np.sqrt(3.0) / 4
    assert np.allclose(a, np.array([0.75, -0.25, -0.25, -0.25]) / s, rtol=1e-6)


def test_equal_rewards_and_singletons_give_zero():
    assert np.all(group_advantage([1, 1, 1, 1, 0, 0, 0, 0], 4, EPS) == 0)
    assert np.all(group_advantage([3.0, -2.0, 7.0], 1, EPS) == 0)


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("unbiased", [True, False])
def test_matches_numpy_std(seed, unbiased):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([2, 4, 8, 16]))
    r = rng.normal(size=G * 6).astype(np.float32)
    a = group_advantage(r, G, EPS, unbiased)
    rr = r.astype(np.float64).reshape(-1, G)
    want = (rr - rr.mean(1, keepdims=True)) / (rr.std(1, ddof=1 if unbiased else 0, keepdims=True) + float(EPS))
    assert np.allclose(a, want.reshape(-1), rtol=2e-7, atol=1e-7)
    # each group's advantages sum to ~0 (centred)
    assert np.allclose(a.reshape(-1, G).astype(np.float64).sum(1), 0, atol=1e-5)


def test_broadcast_pad_rows_zero():
    tok = broadcast_to_tokens(np.array([0.5, -1.0], np.float32), [0, 1, -1, 1], [2, 1, 3, 2])
    assert tok.tolist() == [0.5, 0.5, -1.0, 0.0, 0.0, 0.0, -1.0, -1.0]
