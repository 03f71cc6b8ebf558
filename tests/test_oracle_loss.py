"""Pins for the oracle loss and gradient: closed forms, scipy, finite differences, invariants.
CPU only."""
import math

import numpy as np
import pytest
import scipy.special as sps

from oracle import loss as L

EPS = 0.2


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4040, 0x0000, 0x8000, 0x7F80, 0x3E80], np.uint16)
    assert L.bf16_bits_to_f64(bits).tolist() == [1.0, -1.0, 3.0, 0.0, -0.0, math.inf, 0.25]


@pytest.mark.parametrize("V", [2, 7, 512, 4096])
def test_log_softmax_matches_scipy(V):
    z = np.random.default_rng(V).normal(0, 3, V)
    assert np.allclose(L.log_softmax_row(z), sps.log_softmax(z), rtol=0, atol=1e-12)


def test_two_token_hand_case():
    # z = [0, 0], y = 0: logp = -ln 2; old = -ln 2 -> r = 1; A = 1 -> l = -1;
    # dz = A * r * (softmax - onehot) = (0.5 - 1, 0.5)
    lt, lp, r, cl, dz = L.token_objective(np.zeros(2), 0, -math.log(2), 1.0, 1, EPS)
    assert lp == pytest.approx(-math.log(2), abs=1e-15)
    assert r == pytest.approx(1.0, abs=1e-15) and not cl
    assert lt == pytest.approx(-1.0, abs=1e-15)
    assert np.allclose(dz, [-0.5, 0.5], atol=1e-15)


@pytest.mark.parametrize("r,A,loss,clipped", [
    (1.5, 2.0, -1.2 * 2.0, True),    # A > 0, r above 1+eps: the clip binds, gradient 0
    (0.5, -2.0, 0.8 * 2.0, True),    # A < 0, r below 1-eps: binds
    (0.5, 2.0, -0.5 * 2.0, False),   # A > 0, r below 1-eps: min picks r*A, gradient flows
    (1.5, -2.0, 1.5 * 2.0, False),   # A < 0, r above 1+eps: min picks r*A, gradient flows
    (1.1, 2.0, -1.1 * 2.0, False),   # inside the trust region
    (1.0, 0.0, 0.0, False),          # zero advantage
])
def test_clip_cases(r, A, loss, clipped):
    z = np.array([0.3, -1.0, 2.0, 0.5])
    y = 2
    logp = float(sps.log_softmax(z)[y])
    old = logp - math.log(r)
    lt, lp, rr, cl, dz = L.token_objective(z, y, old, A, 1, EPS)
    assert rr == pytest.approx(r, rel=1e-12)
    assert lt == pytest.approx(loss, rel=1e-12, abs=1e-15)
    assert cl == clipped
    if clipped or A == 0:
        assert np.all(dz == 0)
    else:
        want = A * r * (sps.softmax(z) - np.eye(4)[y])
        assert np.allclose(dz, want, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_ratio_one_closed_form(seed):
    # no pi_old (pi_old = current policy): r = exp(0) = 1, the clip never binds, so
    # loss = -sum(m * A) / N and dz = A * (softmax - onehot) / N.
    rng = np.random.default_rng(seed)
    T, V = 12, 33
    z = rng.normal(0, 2, (T, V))
    y = rng.integers(0, V, T)
    A = rng.normal(size=T)
    m = (rng.random(T) < 0.7).astype(np.uint8)
    N = int(m.sum())
    out = L.loss_fwd_bwd(z, y, None, A, m, EPS, scale=1.0 / max(N, 1))
    fin = L.finish_step(out["loss_tok"], m, out["clipped"])
    assert fin["loss"] == pytest.approx(-float(np.sum(m * A)) / max(N, 1), rel=1e-13)
    sm = sps.softmax(z, axis=1)
    want = (m * A)[:, None] * (sm - np.eye(V)[y]) / max(N, 1)
    assert np.allclose(out["dlogits"], want, rtol=1e-12, atol=1e-16)
    assert fin["n_clipped"] == 0


def _loss_of(z, y, old, A, m):
    N = max(int(np.sum(m)), 1)
    s = 0.0
    for t in range(z.shape[0]):
        lt, *_ = L.token_objective(z[t], int(y[t]), old[t], A[t], int(m[t]), EPS, want_grad=False)
        s += lt
    return s / N


@pytest.mark.parametrize("V", [4, 8, 16])
@pytest.mark.parametrize("seed", range(3))
def test_gradient_central_differences(V, seed):
    rng = np.random.default_rng(100 * V + seed)
    T = 8
    z = rng.normal(0, 1.5, (T, V))
    y = rng.integers(0, V, T)
    A = rng.choice([-1.3, -0.4, 0.7, 1.9], T)
    lsm = np.array([sps.log_softmax(z[t])[y[t]] for t in range(T)])
    # ratios spread over all clip regions, kept 1e-2 away from the kinks at 1 +- eps
    r = rng.choice([0.5, 0.7, 0.95, 1.05, 1.15, 1.3, 1.6], T)
    old = lsm - np.log(r)
    m = np.ones(T, np.uint8)
    m[rng.integers(0, T)] = 0
    N = int(m.sum())
    out = L.loss_fwd_bwd(z, y, old, A, m, EPS, scale=1.0 / N)
    h = 1e-6
    fd = np.zeros_like(z)
    for t in range(T):
        for v in range(V):
            zp = z.copy(); zp[t, v] += h
            zm = z.copy(); zm[t, v] -= h
            fd[t, v] = (_loss_of(zp, y, old, A, m) - _loss_of(zm, y, old, A, m)) / (2 * h)
    assert np.allclose(out["dlogits"], fd, rtol=1e-5, atol=1e-8)
    # dlogits rows sum to zero (softmax sums to one, the one-hot too)
    assert np.allclose(out["dlogits"].sum(1), 0, atol=1e-15)


def test_padding_rows_contribute_nothing():
    rng = np.random.default_rng(7)
    T, V = 10, 16
    z = rng.normal(0, 2, (T, V))
    y = rng.integers(0, V, T)
    A = rng.normal(size=T)
    old = rng.normal(-3, 0.1, T)
    m = np.ones(T, np.uint8)
    base = L.loss_fwd_bwd(z, y, old, A, m, EPS, scale=1.0)
    # append padding rows (copies of a real row's input, mask 0, advantage 0)
    z2 = np.vstack([z, z[:3]])
    y2 = np.concatenate([y, y[:3]])
    A2 = np.concatenate([A, np.zeros(3)])
    old2 = np.concatenate([old, old[:3]])
    m2 = np.concatenate([m, np.zeros(3, np.uint8)])
    pad = L.loss_fwd_bwd(z2, y2, old2, A2, m2, EPS, scale=1.0)
    assert np.array_equal(pad["loss_tok"][:T], base["loss_tok"])
    assert np.all(pad["loss_tok"][T:] == 0) and np.all(pad["dlogits"][T:] == 0)
    assert L.finish_step(pad["loss_tok"], m2)["loss"] == L.finish_step(base["loss_tok"], m)["loss"]


def test_deferred_normalisation_linearity():
    # sum over chunks of the un-normalised chunk gradients, divided once by N, equals the
    # gradient of the un-chunked token mean (gradients are linear)
    rng = np.random.default_rng(11)
    T, V = 12, 20
    z = rng.normal(0, 2, (T, V))
    y = rng.integers(0, V, T)
    A = rng.normal(size=T)
    old = np.array([sps.log_softmax(z[t])[y[t]] for t in range(T)]) + rng.normal(0, 0.05, T)
    m = (rng.random(T) < 0.8).astype(np.uint8)
    N = int(m.sum())
    whole = L.loss_fwd_bwd(z, y, old, A, m, EPS, scale=1.0 / N)
    parts = []
    for a, b in [(0, 5), (5, 6), (6, 12)]:
        parts.append(L.loss_fwd_bwd(z[a:b], y[a:b], old[a:b], A[a:b], m[a:b], EPS, scale=1.0)["dlogits"])
    deferred = np.vstack(parts) / max(N, 1)
    assert np.allclose(deferred, whole["dlogits"], rtol=1e-14, atol=1e-18)
    # a mean of chunk means differs on unequal chunks (the bug the pages warn about)
    lt = whole["loss_tok"]
    mom = np.mean([lt[a:b].sum() / max(m[a:b].sum(), 1) for a, b in [(0, 5), (5, 6), (6, 12)]])
    assert abs(mom - lt.sum() / N) > 1e-6


def test_all_empty_step_is_zero_not_nan():
    fin = L.finish_step(np.zeros(5), np.zeros(5, np.uint8))
    assert fin["loss"] == 0.0 and fin["n_valid"] == 0


def test_lmhead_oracle_matches_chain_rule():
    # d_h and dW follow from dlogits by the chain rule of z = h W^T; pinned by central
    # differences of the step loss with respect to h and W on a tiny problem
    rng = np.random.default_rng(31)
    T, H, V = 5, 6, 7
    h = rng.normal(0, 1, (T, H))
    W = rng.normal(0, 0.5, (V, H))
    y = rng.integers(0, V, T)
    A = rng.choice([-1.0, 0.5, 2.0], T)
    m = np.array([1, 1, 0, 1, 1], np.uint8)
    z = h @ W.T
    lsm = np.array([sps.log_softmax(z[t])[y[t]] for t in range(T)])
    old = lsm - np.log(rng.choice([0.9, 1.05, 1.1], T))
    N = int(m.sum())
    out = L.lmhead_fwd_bwd(h, W, y, old, A, m, EPS, scale=1.0 / N)

    def f(hh, WW):
        zz = hh @ WW.T
        return sum(L.token_objective(zz[t], int(y[t]), old[t], A[t], int(m[t]), EPS, want_grad=False)[0]
                   for t in range(T)) / N

    eps_fd = 1e-6
    for (i, j) in [(0, 0), (1, 3), (4, 5), (3, 2)]:
        hp, hm = h.copy(), h.copy()
        hp[i, j] += eps_fd
        hm[i, j] -= eps_fd
        assert out["d_h"][i, j] == pytest.approx((f(hp, W) - f(hm, W)) / (2 * eps_fd), rel=1e-5, abs=1e-9)
    for (i, j) in [(0, 0), (6, 5), (3, 1), (2, 4)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[i, j] += eps_fd
        Wm[i, j] -= eps_fd
        assert out["dW"][i, j] == pytest.approx((f(h, Wp) - f(h, Wm)) / (2 * eps_fd), rel=1e-5, abs=1e-9)
    # the vocabulary sum of dW vanishes (each dlogits row sums to zero)
    assert np.allclose(out["dW"].sum(0), 0, atol=1e-12)
    # the masked token's hidden row gets no gradient
    assert np.all(out["d_h"][2] == 0)


@pytest.mark.parametrize("kind, ent", [(2, 0.0), (0, 0.05), (1, 0.03)])
def test_lmhead_oracle_with_terms_matches_chain_rule(kind, ent):
    # the LM-head oracle with the regularisers (KL k1/k3 to a reference policy, the entropy
    # bonus) and per-token gradient weights: d_h and dW are the central differences of the
    # weighted step loss sum_t w_t l_t / N with respect to h and W
    rng = np.random.default_rng(60 + kind)
    T, H, V = 5, 6, 7
    h = rng.normal(0, 1, (T, H))
    W = rng.normal(0, 0.5, (V, H))
    y = rng.integers(0, V, T)
    A = rng.choice([-1.0, 0.5, 2.0], T)
    m = np.array([1, 1, 0, 1, 1], np.uint8)
    z = h @ W.T
    lsm = np.array([sps.log_softmax(z[t])[y[t]] for t in range(T)])
    old = lsm - np.log(rng.choice([0.9, 1.05, 1.1], T))
    ref = lsm + rng.normal(0, 0.3, T)
    w = rng.choice([1.0, 0.5, 0.25], T)
    N = int(m.sum())
    terms = dict(kl_kind=kind, kl_coef=0.1, ref=ref, ent_coef=ent)
    out = L.lmhead_fwd_bwd(h, W, y, old, A, m, EPS, scale=w / N, terms=terms)

    def f(hh, WW):
        zz = hh @ WW.T
        tot = 0.0
        for t in range(T):
            tt = dict(kl_kind=kind, kl_coef=0.1, ref=ref[t], ent_coef=ent)
            tot += w[t] * L.token_objective(zz[t], int(y[t]), old[t], A[t], int(m[t]), EPS, want_grad=False,
                                            terms=tt)[0]
        return tot / N

    eps_fd = 1e-6
    for (i, j) in [(0, 0), (1, 3), (4, 5), (3, 2)]:
        hp, hm = h.copy(), h.copy()
        hp[i, j] += eps_fd
        hm[i, j] -= eps_fd
        assert out["d_h"][i, j] == pytest.approx((f(hp, W) - f(hm, W)) / (2 * eps_fd), rel=1e-5, abs=1e-9)
    for (i, j) in [(0, 0), (6, 5), (3, 1), (2, 4)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[i, j] += eps_fd
        Wm[i, j] -= eps_fd
        assert out["dW"][i, j] == pytest.approx((f(h, Wp) - f(h, Wm)) / (2 * eps_fd), rel=1e-5, abs=1e-9)
    assert np.all(out["d_h"][2] == 0)


@pytest.mark.parametrize("kind", [1, 2])
@pytest.mark.parametrize("ent", [0.0, 0.03])
def test_extra_terms_central_differences(kind, ent):
    # KL to a reference policy (k1 or k3) and an entropy bonus: the analytic dlogits equal
    # central differences of the per-token loss; the entropy equals scipy's
    rng = np.random.default_rng(40 + kind)
    V = 9
    for _ in range(4):
        z = rng.normal(0, 1.5, V)
        y = int(rng.integers(0, V))
        lsm = sps.log_softmax(z)
        old = lsm[y] - math.log(rng.choice([0.9, 1.05]))
        A = float(rng.choice([-1.0, 0.7]))
        terms = dict(kl_kind=kind, kl_coef=0.1, ref=lsm[y] + rng.normal(0, 0.3), ent_coef=ent)
        lt, lp, r, cl, dz = L.token_objective(z, y, old, A, 1, EPS, 1.0, True, dict(terms))
        t2 = dict(terms)
        L.token_objective(z, y, old, A, 1, EPS, 1.0, False, t2)
        p = sps.softmax(z)
        assert t2["entropy"] == pytest.approx(-float(np.sum(p * np.log(p))), rel=1e-12)
        h = 1e-6
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[v] += h
            zm[v] -= h
            fp = L.token_objective(zp, y, old, A, 1, EPS, 1.0, False, dict(terms))[0]
            fm = L.token_objective(zm, y, old, A, 1, EPS, 1.0, False, dict(terms))[0]
            assert dz[v] == pytest.approx((fp - fm) / (2 * h), rel=1e-5, abs=1e-9)


def test_k3_is_zero_at_the_reference_and_nonnegative():
    z = np.array([0.5, -1.0, 2.0])
    lp = float(sps.log_softmax(z)[2])
    t = dict(kl_kind=2, kl_coef=1.0, ref=lp)
    base = L.token_objective(z, 2, lp, 0.0, 1, EPS)[0]
    assert L.token_objective(z, 2, lp, 0.0, 1, EPS, terms=t)[0] == pytest.approx(base, abs=1e-15)
    for ref in (lp - 1.0, lp + 0.5):
        t = dict(kl_kind=2, kl_coef=1.0, ref=ref)
        assert L.token_objective(z, 2, lp, 0.0, 1, EPS, terms=t)[0] >= base


def test_entropy_ignores_masked_vocabulary_entries():
    # a -inf logit has no mass: the entropy and its gradient equal those of the row without it
    z = np.array([0.3, -np.inf, 1.2, -0.7])
    zr = np.array([0.3, 1.2, -0.7])
    t1, t2 = dict(ent_coef=0.1), dict(ent_coef=0.1)
    l1, _, _, _, d1 = L.token_objective(z, 2, None, 0.5, 1, EPS, 1.0, True, t1)
    l2, _, _, _, d2 = L.token_objective(zr, 1, None, 0.5, 1, EPS, 1.0, True, t2)
    assert t1["entropy"] == pytest.approx(t2["entropy"], rel=1e-14)
    assert l1 == pytest.approx(l2, rel=1e-14)
    assert d1[1] == 0 and np.allclose(np.delete(d1, 1), d2, rtol=1e-13)


@pytest.mark.parametrize("c", [1e3, -4e3, 2.0 ** 40, -(2.0 ** 44)])
def test_objective_is_shift_invariant(c):
    # log-softmax, and so the whole token objective and its gradient, does not change when a
    # constant is added to a row. With logits on a 2^-8 grid and shifts that keep them exact in
    # float64 (up to 2^44), the oracle gives the same numbers at any offset: it subtracts the
    # row maximum before exponentiating. The library's shift-invariance test compares with it.
    rng = np.random.default_rng(11)
    z = np.round(rng.normal(0, 3.0, 64) * 256) / 256
    zc = z + c
    assert np.array_equal(zc - c, z)
    base = L.token_objective(z, 5, -2.0, 0.7, 1, 0.2, 1.0 / 7, True)
    shifted = L.token_objective(zc, 5, -2.0, 0.7, 1, 0.2, 1.0 / 7, True)
    for a, b in zip(base[:3], shifted[:3]):  # loss, log-prob, ratio
        assert abs(a - b) <= 1e-12 * max(1.0, abs(a))
    assert base[3] == shifted[3]  # the clip decision
    assert np.allclose(base[4], shifted[4], rtol=1e-12, atol=1e-15)
