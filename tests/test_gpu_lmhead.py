"""GPU parity of the fused LM-head variant (tcgen05 GEMMs + softmax epilogue) against the
float64 oracle: per-token loss and log-prob, d_h and dW, on sizes with ragged token, vocabulary
and K tiles, several vocabulary chunks, masked tokens and forward-only calls, for both tile
shapes (the paired 2-CTA MMA of the product path and the one-CTA instance).

d_h and dW tolerance: both products are formed from bf16 dlogits (rounded to nearest), so
each element may move by up to ~2^-8 of the sum of the magnitudes of its terms; the bar is
|d| <= 8e-3 * (|dz| |W|)_ij (resp. (|dz|^T |h|)_ij) + 1e-12."""
import numpy as np
import pytest
import torch

from oracle import advantage as OA
from oracle import loss as OL
from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import workloads as W

from tests import _gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built(grpo_lib):
    assert torch.cuda.is_available()
    return grpo_lib


@pytest.fixture(params=[2, 1], ids=["pair", "one_cta"])
def cta_group(request, monkeypatch):
    """Tile shape of the LM-head GEMMs (read by the library on every call)."""
    monkeypatch.setenv("GRPO_LMHEAD_CTA_GROUP", str(request.param))
    return request.param


def _case(T, V, Hd, seed, valid_lo=None, old=True, adv=None, w_row_scale=None):
    wl = W.make_workload("lmhead", seed=seed, rows=4, tokens=T, V=V, H=Hd)
    assert wl.T == T, (wl.T, T)
    h, Wt = W.make_lmhead_inputs(wl, DEV)
    if w_row_scale is not None:  # (rows, factor): a few vocabulary entries with much larger logits
        rows, factor = w_row_scale
        Wt[rows] = (Wt[rows].float() * factor).to(torch.bfloat16)
    hb = h.view(torch.int16).cpu().numpy().view(np.uint16)
    wb = Wt.view(torch.int16).cpu().numpy().view(np.uint16)
    mask = wl.mask.copy()
    if valid_lo is not None:
        mask[np.random.default_rng(seed).random(T) < valid_lo] = 0
    a_tok = OA.broadcast_to_tokens(OA.group_advantage(wl.rewards, wl.group_size, np.float32(1e-6)),
                                   wl.row_rollout, wl.row_len) if adv is None else adv.astype(np.float32)
    old_logp = None
    if old:
        z = OL.as_f64(hb) @ OL.as_f64(wb).T
        ref = np.array([OL.log_softmax_row(z[t])[wl.target[t]] for t in range(T)])
        old_logp = (ref + wl.old_noise).astype(np.float32)
    return wl, h, Wt, hb, wb, mask, a_tok, old_logp


def _run(h, Wt, wl, mask, a_tok, old_logp, scale, grads=True):
    T, Hd = h.shape
    V = Wt.shape[0]
    d_h = torch.full((T, Hd), 7.0, device=DEV) if grads else None
    dW = torch.full((V, Hd), 7.0, device=DEV) if grads else None
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, scale,
                                  d_h, dW, loss, logp, acc, ws)
    torch.cuda.synchronize()
    return d_h, dW, loss, logp, acc


def _check(T, V, Hd, seed, valid_lo=None, old=True, adv=None, grads=True, w_row_scale=None):
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed, valid_lo, old, adv, w_row_scale)
    N = max(int(mask.sum()), 1)
    d_h, dW, loss, logp, acc = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / N, grads)
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=1.0 / N)
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, a_tok, mask)
    res = _lib.grpo_finish_step(acc, loss, expected_N=int(mask.sum()))
    assert res["status"] == 0 and res["kernel_flags"] == 0
    if not grads:
        return ref
    # tolerance from the magnitudes of the terms of each product
    hf, wf = OL.as_f64(hb), OL.as_f64(wb)
    z = hf @ wf.T
    dz_abs = np.zeros_like(z)
    for t in range(T):
        if mask[t]:
            dz_abs[t] = np.abs(OL.token_objective(z[t], int(wl.target[t]), None if old_logp is None else old_logp[t],
                                                  a_tok[t], 1, wl.eps, 1.0 / N)[4])
    tol_h = 8e-3 * (dz_abs @ np.abs(wf)) + 1e-12
    tol_w = 8e-3 * (dz_abs.T @ np.abs(hf)) + 1e-12
    gh, gw = H.to_f64(d_h), H.to_f64(dW)
    bad_h = np.abs(gh - ref["d_h"]) > tol_h
    bad_w = np.abs(gw - ref["dW"]) > tol_w
    assert not bad_h.any(), (np.argwhere(bad_h)[:3], gh[bad_h][:3], ref["d_h"][bad_h][:3])
    assert not bad_w.any(), (np.argwhere(bad_w)[:3], gw[bad_w][:3], ref["dW"][bad_w][:3])
    return ref


def test_lmhead_exact_tiles(cta_group):
    _check(256, 1024, 128, seed=1)


def test_lmhead_ragged_tokens_vocab_and_k(cta_group):
    # 300 tokens (ragged 128-row and 256-row tiles), V = 1000 (ragged 256-column tile and
    # 32-column group), H = 192 (three 64-wide K blocks; a d_h / dW column tile of 192 of 256)
    _check(300, 1000, 192, seed=2)


def test_lmhead_several_vocab_chunks_masked_tokens(cta_group):
    # V = 40000: 157 vocabulary tiles in three chunks of 53 (the last ragged), so d_h is
    # accumulated over three chunk products; a quarter of the tokens masked
    _check(128, 40000, 64, seed=3, valid_lo=0.25)


def test_lmhead_no_pi_old_and_clip_stress(cta_group):
    T = 256
    adv = np.random.default_rng(4).choice([-2.0, -0.5, 0.5, 2.0], T)
    _check(T, 2048, 128, seed=4, old=False, adv=adv)


def test_lmhead_wide_logit_spread(cta_group):
    # columns 300..307 get logits ~300x larger than the rest (a spread far beyond 2^64 in the
    # exponent): the partials' lazy shift must rescale instead of overflowing
    _check(256, 1024, 128, seed=6, w_row_scale=(slice(300, 308), 300.0))


def test_lmhead_forward_only(cta_group):
    _check(256, 4096, 256, seed=5, grads=False)


def test_lmhead_product_vocabulary_full_oracle(cta_group):
    # the product vocabulary and hidden size (V = 151936, H = 2048) at 512 tokens, where the
    # float64 oracle forms every logit: per-token outputs on every token, d_h on every row and
    # dW on 300 sampled vocabulary rows plus every row some token targets, elementwise
    T, V, Hd = 512, 151936, 2048
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=11, valid_lo=0.1)
    N = max(int(mask.sum()), 1)
    d_h, dW, loss, logp, acc = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / N)
    res = _lib.grpo_finish_step(acc, loss, expected_N=int(mask.sum()))
    assert res["status"] == 0 and res["kernel_flags"] == 0
    hf, wf = OL.as_f64(hb), OL.as_f64(wb)
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=1.0 / N, want_dw=False)
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, a_tok, mask)
    z = hf @ wf.T
    dz = np.zeros_like(z)
    for t in range(T):
        if mask[t]:
            dz[t] = OL.token_objective(z[t], int(wl.target[t]), old_logp[t], a_tok[t], 1, wl.eps, 1.0 / N)[4]
    del z
    dz_abs = np.abs(dz)
    tol_h = 8e-3 * (dz_abs @ np.abs(wf)) + 1e-12
    gh = H.to_f64(d_h)
    bad = np.abs(gh - ref["d_h"]) > tol_h
    assert not bad.any(), (np.argwhere(bad)[:3], gh[bad][:3], ref["d_h"][bad][:3])
    rows = np.unique(np.concatenate([np.random.default_rng(12).choice(V, 300, replace=False),
                                     wl.target[mask.astype(bool)], [0, V - 1]]))
    want = dz[:, rows].T @ hf
    tol_w = 8e-3 * (dz_abs[:, rows].T @ np.abs(hf)) + 1e-12
    gw = dW[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    bad = np.abs(gw - want) > tol_w
    assert not bad.any(), (rows[np.argwhere(bad)[:3, 0]], gw[bad][:3], want[bad][:3])


def test_lmhead_full_size_sampled_rows():
    # the full fused LM-head shape (16384 tokens, H = 2048, V = 151936) in the bench's launch
    # configuration; per-token outputs and d_h checked on sampled rows (the oracle recomputes
    # those rows' logits one by one), dW checked by a property that holds at any size: every
    # dlogits row sums to zero, so the vocabulary sum of dW vanishes
    wl = W.make_workload("lmhead", seed=0)
    T, V, Hd = wl.T, wl.V, wl.extra["H"]
    h, Wt = W.make_lmhead_inputs(wl, DEV)
    adv = np.random.default_rng(9).choice([-1.5, -0.3, 0.4, 1.2], T).astype(np.float32)
    N = int(wl.mask.sum())
    d_h, dW, loss, logp, acc = _run(h, Wt, wl, wl.mask, adv, None, 1.0 / N)
    res = _lib.grpo_finish_step(acc, loss, expected_N=N)
    assert res["status"] == 0 and res["n_valid"] == N and res["kernel_flags"] == 0
    rows = np.array([0, 1, 127, 128, 255, 256, 5000, 9999, 16254, 16383])
    hb = h[torch.from_numpy(rows).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
    wb = Wt.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target[rows], None, adv[rows], wl.mask[rows], wl.eps,
                            scale=1.0 / N, want_dw=False)
    H.assert_tokens_close(H.to_f64(loss)[rows], H.to_f64(logp)[rows], ref, adv[rows], wl.mask[rows])
    wf = OL.as_f64(wb)
    z = OL.as_f64(hb) @ wf.T
    for k, t in enumerate(rows):
        dz = np.abs(OL.token_objective(z[k], int(wl.target[t]), None, adv[t], 1, wl.eps, 1.0 / N)[4])
        tol = 8e-3 * (dz @ np.abs(wf)) + 1e-12
        got = d_h[int(t)].double().cpu().numpy()
        assert np.all(np.abs(got - ref["d_h"][k]) <= tol), int(t)
    col = dW.double().sum(0)
    mag = dW.double().abs().sum(0)
    assert torch.all(col.abs() <= 2e-2 * mag + 1e-9)
    assert torch.isfinite(dW).all() and torch.isfinite(d_h).all()


def test_lmhead_tile_shapes_agree():
    # the paired 256 x 256 tiles and the one-CTA 128 x 256 tiles sum every product in the same
    # K order: identical bits for every output
    T, V, Hd = 300, 5000, 192
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=21, valid_lo=0.2)
    outs = []
    for cg in (2, 1):
        import os
        os.environ["GRPO_LMHEAD_CTA_GROUP"] = str(cg)
        try:
            outs.append(_run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / max(int(mask.sum()), 1)))
        finally:
            del os.environ["GRPO_LMHEAD_CTA_GROUP"]
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert torch.equal(a, b)


def _oracle_grad_tol(hb, wb, wl, mask, a_tok, old_logp, N):
    """The oracle's d_h and dW for a case, and the elementwise bars of the module docstring."""
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=1.0 / N)
    hf, wf = OL.as_f64(hb), OL.as_f64(wb)
    z = hf @ wf.T
    dz_abs = np.zeros_like(z)
    for t in range(z.shape[0]):
        if mask[t]:
            dz_abs[t] = np.abs(OL.token_objective(z[t], int(wl.target[t]), None if old_logp is None else old_logp[t],
                                                  a_tok[t], 1, wl.eps, 1.0 / N)[4])
    return ref, 8e-3 * (dz_abs @ np.abs(wf)) + 1e-12, 8e-3 * (dz_abs.T @ np.abs(hf)) + 1e-12


@pytest.mark.parametrize("deferred", [False, True])
def test_lmhead_micro_batches_accumulate_dw(cta_group, deferred):
    # one optimizer step as three micro-batches (token blocks of 128, 200 and 172: ragged tiles),
    # one call each with dW accumulated ("Sizing mini-batches and micro-batches", "The hard part:
    # deferred normalization"), at the step's grad scale 1/N or, deferred, at 1 with the finish
    # scaling d_h and dW once. Per-token outputs and the step loss equal the one-call step's;
    # d_h and dW (the sum of three float32 products) meet the oracle's bar.
    T, V, Hd = 500, 3000, 128
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=31, valid_lo=0.1)
    N = max(int(mask.sum()), 1)
    one = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / N)
    res_one = _lib.grpo_finish_step(one[4], one[2], expected_N=int(mask.sum()))
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d_h = torch.full((T, Hd), 7.0, device=DEV)
    dW = torch.full((V, Hd), 7.0, device=DEV)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    bounds = [0, 128, 328, 500]
    for k in range(3):
        a, b = bounds[k], bounds[k + 1]
        ws = torch.empty(_lib.grpo_lmhead_workspace_size(b - a, V, Hd), dtype=torch.uint8, device=DEV)
        _lib.grpo_lmhead_loss_fwd_bwd(h[a:b], Wt, t(wl.target[a:b]), t(old_logp[a:b]), t(a_tok[a:b]), t(mask[a:b]),
                                      wl.eps, 1.0 if deferred else 1.0 / N, d_h[a:b], dW, loss[a:b], logp[a:b],
                                      acc, ws, dw_accumulate=k > 0)
    res = _lib.grpo_finish_step(acc, loss, expected_N=int(mask.sum()), deferred=deferred, grad_bufs=[d_h, dW])
    torch.cuda.synchronize()
    assert res["status"] == 0 and res["kernel_flags"] == 0
    for key in ("loss", "n_valid", "n_clipped", "n_tokens"):
        assert res[key] == res_one[key], key
    assert torch.equal(loss, one[2]) and torch.equal(logp, one[3])
    if not deferred:
        # a token's d_h row depends on that token alone: the same bits in any micro-batch
        assert torch.equal(d_h, one[0])
    ref, tol_h, tol_w = _oracle_grad_tol(hb, wb, wl, mask, a_tok, old_logp, N)
    gh, gw = H.to_f64(d_h), H.to_f64(dW)
    bad = np.abs(gh - ref["d_h"]) > tol_h
    assert not bad.any(), (np.argwhere(bad)[:3], gh[bad][:3], ref["d_h"][bad][:3])
    bad = np.abs(gw - ref["dW"]) > tol_w
    assert not bad.any(), (np.argwhere(bad)[:3], gw[bad][:3], ref["dW"][bad][:3])


@pytest.mark.parametrize("T, V, Hd", [(1, 1, 64), (3, 300, 64), (129, 257, 64), (2, 40000, 64)])
def test_lmhead_degenerate_sizes(cta_group, T, V, Hd):
    # one token, a one-entry vocabulary (log p = 0, every dlogit 0), tiles that are one row or
    # one column past a multiple of the tile, and a few tokens over several vocabulary chunks
    _check(T, V, Hd, seed=40 + T)


@pytest.mark.parametrize("skip_masked", [False, True])
def test_lmhead_step_captured_in_a_cuda_graph_replays_bitwise(skip_masked):
    # the LM-head step (one call with d_h and dW, then the finish) captured once into a CUDA
    # graph: a replay gives the eager call's bits, and after new hidden states and advantages
    # are written into the same buffers (so the count of tokens with a gradient, read on the
    # device, changes) the replay gives what an eager call on them gives
    T, V, Hd = 300, 5000, 128
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=51)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    tgt, old, adv, msk = t(wl.target), t(old_logp), t(a_tok), t(mask)
    d_h = torch.empty((T, Hd), device=DEV)
    dW = torch.empty((V, Hd), device=DEV)
    loss, logp = torch.empty(T, device=DEV), torch.empty(T, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    N = int(mask.sum())

    def step():
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, tgt, old, adv, msk, wl.eps, 1.0 / max(N, 1), d_h, dW, loss, logp,
                                      acc, ws, skip_masked=skip_masked)
        _lib.grpo_finish_step(acc, loss, expected_N=N, sync=False)

    def snapshot():
        torch.cuda.synchronize()
        return d_h.clone(), dW.clone(), loss.clone(), logp.clone(), acc[64:128].clone()

    step()  # eager (sets the kernels' attributes before the capture)
    eager = snapshot()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            step()
    for _ in range(2):
        d_h.fill_(7.0)
        dW.fill_(7.0)
        g.replay()
        for a, b in zip(snapshot(), eager):
            assert torch.equal(a, b)
    h.copy_(torch.flip(h, dims=[0]))
    adv.copy_(torch.where(torch.arange(T, device=DEV) % 5 < 2, torch.zeros_like(adv), adv))
    g.replay()
    replayed = snapshot()
    step()
    for a, b in zip(replayed, snapshot()):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[0], eager[0])


@pytest.mark.parametrize("deferred", [False, True])
def test_lmhead_nonfinite_hidden_state_skips_the_step(deferred):
    # a NaN planted in one token's hidden state (host-side fault injection): that token's
    # logits, log-prob and loss are not finite, the finish reports the step skipped and zeroes
    # the gradient buffers it is given (d_h and dW), and every other token's outputs still match
    # the oracle
    T, V, Hd = 200, 3000, 128
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=71)
    bad = 37
    mask[bad] = 1
    h[bad, 5] = float("nan")
    N = int(mask.sum())
    d_h, dW, loss, logp, acc = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 if deferred else 1.0 / N)
    res = _lib.grpo_finish_step(acc, loss, expected_N=N, deferred=deferred, grad_bufs=[d_h, dW])
    assert res["status"] == _lib.STEP_SKIPPED_NONFINITE and res["n_nonfinite"] == 1
    assert res["kernel_flags"] == 0 and res["n_valid"] == N
    assert torch.count_nonzero(d_h) == 0 and torch.count_nonzero(dW) == 0
    gl, gp = H.to_f64(loss), H.to_f64(logp)
    assert not np.isfinite(gp[bad])
    keep = np.ones(T, bool)
    keep[bad] = False
    hb2 = h.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = OL.lmhead_fwd_bwd(hb2[keep], wb, wl.target[keep], old_logp[keep], a_tok[keep], mask[keep], wl.eps,
                            scale=1.0 / N, want_dw=False)
    H.assert_tokens_close(gl[keep], gp[keep], ref, a_tok[keep], mask[keep])


def test_lmhead_backward_overlap_gives_the_same_bits(monkeypatch):
    # the backward's d_h and dW on the library's second stream beside the next chunk's
    # recompute (two chunk buffers) against every launch on the caller's stream: the same bits
    # for every output, over four vocabulary chunks, with dW accumulated into a second call's
    T, V, Hd = 300, 60000, 128
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=81, valid_lo=0.2)
    outs = []
    for ov in ("0", "1"):
        monkeypatch.setenv("GRPO_LMHEAD_OVERLAP", ov)
        d_h, dW, loss, logp, acc = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / max(int(mask.sum()), 1))
        ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, 0.5, d_h, dW,
                                      loss, logp, _lib.new_step_acc(DEV), ws, dw_accumulate=True)
        torch.cuda.synchronize()
        outs.append((d_h, dW, loss, logp))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ---- regularisers through the LM-head: KL to the reference policy, the entropy bonus, and
# per-token gradient weights (grpo_lmhead_loss_fwd_bwd_ex) -------------------------------------

@pytest.mark.parametrize("kl_kind, ent, weighted", [(1, 0.0, False), (2, 0.0, True), (0, 0.05, False),
                                                     (2, 0.02, True)])
def test_lmhead_kl_entropy_and_token_weights(cta_group, kl_kind, ent, weighted):
    # 300 tokens (ragged tiles), V = 20000 (two vocabulary chunks, the second ragged), H = 192;
    # the reference log-probs a normal perturbation of the policy's own, the weights those of
    # sequence-mean aggregation (1 / row length, a few distinct values)
    T, V, Hd = 300, 20000, 192
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=70 + kl_kind, valid_lo=0.1)
    rng = np.random.default_rng(71)
    ref = (old_logp + rng.normal(0, 0.3, T)).astype(np.float32)
    w_tok = rng.choice([1.0, 0.5, 0.125, 1.0 / 3], T).astype(np.float32) if weighted else None
    N = max(int(mask.sum()), 1)
    gs = np.float32(1.0 / N)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d_h = torch.full((T, Hd), 7.0, device=DEV)
    dW = torch.full((V, Hd), 7.0, device=DEV)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    ent_t = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    terms = dict(kl_kind=kl_kind, kl_coef=0.1, ref_logp=t(ref), ent_coef=ent, entropy_tok=ent_t, w_tok=t(w_tok))
    _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, float(gs),
                                  d_h, dW, loss, logp, acc, ws, terms=terms)
    torch.cuda.synchronize()
    # the oracle's per-token scale: the float32 product the kernels form, held in float64
    scale = (gs * w_tok).astype(np.float64) if weighted else float(gs)
    oterms = dict(kl_kind=kl_kind, kl_coef=float(np.float32(0.1)), ref=ref.astype(np.float64),
                  ent_coef=float(np.float32(ent)))
    out = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=scale, terms=oterms)
    m = mask.astype(bool)
    gl, gp, ge = H.to_f64(loss), H.to_f64(logp), H.to_f64(ent_t)
    assert np.all(np.abs(gp[m] - out["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(out["logp_tok"][m])))
    assert np.all(np.abs(ge[m] - out["entropy"][m]) <= 1e-5 * np.maximum(1, out["entropy"][m]))
    assert np.all(ge[~m] == 0) and np.all(gl[~m] == 0) and np.all(gp[~m] == 0)
    assert np.all(np.abs(gl - out["loss_tok"]) <= 1e-5 * np.abs(out["loss_tok"]) + 1e-6)
    res = _lib.grpo_finish_step(acc, loss, expected_N=int(mask.sum()))
    assert res["status"] == 0 and res["kernel_flags"] == 0 and res["n_valid"] == int(mask.sum())
    # d_h and dW: the module docstring's bar over the magnitudes of the regularised dlogits
    hf, wf = OL.as_f64(hb), OL.as_f64(wb)
    z = hf @ wf.T
    dz_abs = np.zeros_like(z)
    for k in range(T):
        if mask[k]:
            tt = dict(oterms, ref=float(ref[k]))
            sk = scale[k] if weighted else scale
            dz_abs[k] = np.abs(OL.token_objective(z[k], int(wl.target[k]), old_logp[k], a_tok[k], 1, wl.eps, sk,
                                                  terms=tt)[4])
    tol_h = 8e-3 * (dz_abs @ np.abs(wf)) + 1e-12
    tol_w = 8e-3 * (dz_abs.T @ np.abs(hf)) + 1e-12
    gh, gw = H.to_f64(d_h), H.to_f64(dW)
    bad = np.abs(gh - out["d_h"]) > tol_h
    assert not bad.any(), (np.argwhere(bad)[:3], gh[bad][:3], out["d_h"][bad][:3])
    bad = np.abs(gw - out["dW"]) > tol_w
    assert not bad.any(), (np.argwhere(bad)[:3], gw[bad][:3], out["dW"][bad][:3])


def test_lmhead_terms_off_gives_the_plain_bits(cta_group):
    # terms with every regulariser off and no per-token outputs take the plain path: the same
    # bits as the call without terms; asking for the entropy as a metric only (ent_coef 0)
    # leaves the loss, log-probs and gradients within the plain call's bars and the entropy at
    # the oracle's
    T, V, Hd = 300, 3000, 128
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=77, valid_lo=0.1)
    N = max(int(mask.sum()), 1)
    plain = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / N)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)

    def run_terms(terms):
        d_h = torch.full((T, Hd), 7.0, device=DEV)
        dW = torch.full((V, Hd), 7.0, device=DEV)
        loss = torch.full((T,), -7.0, device=DEV)
        logp = torch.full((T,), -7.0, device=DEV)
        acc = _lib.new_step_acc(DEV)
        ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, 1.0 / N,
                                      d_h, dW, loss, logp, acc, ws, terms=terms)
        torch.cuda.synchronize()
        return d_h, dW, loss, logp, acc

    off = run_terms(dict(kl_kind=0, kl_coef=0.0, ent_coef=0.0))
    for a, b in zip(plain[:4], off[:4]):
        assert torch.equal(a, b)
    ent_t = torch.full((T,), -7.0, device=DEV)
    met = run_terms(dict(ent_coef=0.0, entropy_tok=ent_t))
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=1.0 / N,
                            terms=dict(kl_kind=0, kl_coef=0.0, ref=None, ent_coef=0.0))
    H.assert_tokens_close(H.to_f64(met[2]), H.to_f64(met[3]), ref, a_tok, mask)
    m = mask.astype(bool)
    ge = H.to_f64(ent_t)
    assert np.all(np.abs(ge[m] - ref["entropy"][m]) <= 1e-5 * np.maximum(1, ref["entropy"][m]))
    assert np.all(ge[~m] == 0)
    _, tol_h, tol_w = _oracle_grad_tol(hb, wb, wl, mask, a_tok, old_logp, N)
    assert not (np.abs(H.to_f64(met[0]) - ref["d_h"]) > tol_h).any()
    assert not (np.abs(H.to_f64(met[1]) - ref["dW"]) > tol_w).any()


def test_lmhead_terms_reject_bad_arguments():
    T, V, Hd = 8, 64, 64
    h = torch.zeros((T, Hd), dtype=torch.bfloat16, device=DEV)
    Wt = torch.zeros((V, Hd), dtype=torch.bfloat16, device=DEV)
    i = torch.zeros(T, dtype=torch.int32, device=DEV)
    f = torch.zeros(T, device=DEV)
    mk = torch.ones(T, dtype=torch.uint8, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    for bad in (dict(kl_kind=7), dict(kl_kind=1)):  # an unknown kind; KL without ref_logp
        with pytest.raises(_lib.GrpoError):
            _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, i, None, f, mk, 0.2, 1.0, None, None, f, None, acc, ws, terms=bad)


# ---- the backward over the live tokens only ---------------------------------------------------
# A token with a zero gradient coefficient (masked, zero advantage, clipped) has an all-zero
# dlogits row; the backward's GEMMs run over the others, in a compact order whose count stays on
# the device. These cases put the count at 0, 1, and just past tile and K-block boundaries.

def _adv_with_live(T, live_rows, seed):
    adv = np.zeros(T, np.float32)
    adv[live_rows] = np.random.default_rng(seed).choice([-1.5, -0.5, 0.5, 1.5], len(live_rows))
    return adv


@pytest.mark.parametrize("n_live", [0, 1, 63, 65, 257])
def test_lmhead_live_token_counts(cta_group, n_live):
    # 600 tokens (ragged), V = 3000, H = 128; the live tokens spread over the call, every other
    # token with a zero advantage; d_h and dW start as 7.0, so a row or entry that no kernel
    # writes fails the comparison
    T, V, Hd = 600, 3000, 128
    live = np.sort(np.random.default_rng(n_live).choice(T, n_live, replace=False))
    adv = _adv_with_live(T, live, seed=80 + n_live)
    ref = _check(T, V, Hd, seed=80, adv=adv)
    assert np.all(ref["d_h"][np.setdiff1d(np.arange(T), live)] == 0)
    if n_live == 0:
        assert np.all(ref["dW"] == 0)


def test_lmhead_dead_tokens_leave_exact_zeros_and_accumulated_dw():
    # every token dead: d_h is written as exact zeros, dW as zeros, and with accumulation dW
    # keeps its bits
    T, V, Hd = 300, 2000, 64
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=90, adv=np.zeros(T))
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d_h = torch.full((T, Hd), 7.0, device=DEV)
    dW = torch.randn((V, Hd), device=DEV)
    dW0 = dW.clone()
    loss = torch.empty(T, device=DEV)
    logp = torch.empty(T, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    args = (h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, 1.0 / T, d_h, dW, loss, logp, acc, ws)
    _lib.grpo_lmhead_loss_fwd_bwd(*args, dw_accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(d_h, torch.zeros_like(d_h))
    assert torch.equal(dW, dW0)
    res = _lib.grpo_finish_step(acc, loss)
    assert res["status"] == 0 and res["n_valid"] == int(mask.sum())
    acc2 = _lib.new_step_acc(DEV)
    _lib.grpo_lmhead_loss_fwd_bwd(*args[:12], acc2, ws)
    torch.cuda.synchronize()
    assert torch.equal(dW, torch.zeros_like(dW))


def test_lmhead_live_tokens_reuse_a_dirty_workspace():
    # the compact hidden-state buffer and the dlogits chunks hold another call's values (and
    # NaN bytes) when a call with fewer live tokens runs: the padded rows it reduces over must
    # be its own zeros
    T, V, Hd = 400, 3000, 128
    ws = torch.full((_lib.grpo_lmhead_workspace_size(T, V, Hd),), 0xFF, dtype=torch.uint8, device=DEV)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    outs = []
    for n_live, seed in ((400, 91), (37, 92)):
        live = np.arange(0, T, T // n_live)[:n_live] if n_live < T else np.arange(T)
        adv = _adv_with_live(T, live, seed=seed)
        wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=93, adv=adv)
        d_h = torch.full((T, Hd), 7.0, device=DEV)
        dW = torch.full((V, Hd), 7.0, device=DEV)
        loss = torch.empty(T, device=DEV)
        logp = torch.empty(T, device=DEV)
        acc = _lib.new_step_acc(DEV)
        N = int(mask.sum())
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, 1.0 / N,
                                      d_h, dW, loss, logp, acc, ws)
        torch.cuda.synchronize()
        ref, tol_h, tol_w = _oracle_grad_tol(hb, wb, wl, mask, a_tok, old_logp, N)
        assert not (np.abs(H.to_f64(d_h) - ref["d_h"]) > tol_h).any()
        assert not (np.abs(H.to_f64(dW) - ref["dW"]) > tol_w).any()
        outs.append((d_h, dW))
    # and the second call's results equal those of the same call on a fresh workspace
    fresh = _run(h, Wt, wl, mask, a_tok, old_logp, 1.0 / N)
    assert torch.equal(outs[1][0], fresh[0]) and torch.equal(outs[1][1], fresh[1])


@pytest.mark.parametrize("with_terms", [False, True], ids=["plain", "kl_entropy_weights"])
def test_lmhead_full_size_bench_configuration(with_terms):
    # the bench's LM-head step at full size (16384 tokens, H = 2048, V = 151936): the group
    # advantages of the workload's rewards (one of its two groups has equal rewards, so half
    # the tokens have no gradient), plain or with KL k3, the entropy bonus and per-token
    # weights. Sampled rows (dead and live ones, tile edges) against the oracle row by row;
    # every d_h row of a token without a gradient exactly zero (plain); dW by the property that
    # every dlogits row sums to zero, so the vocabulary sum of dW vanishes
    wl = W.make_workload("lmhead", seed=0)
    T, V, Hd = wl.T, wl.V, wl.extra["H"]
    h, Wt = W.make_lmhead_inputs(wl, DEV)
    adv = OA.broadcast_to_tokens(OA.group_advantage(wl.rewards, wl.group_size, np.float32(1e-6)),
                                 wl.row_rollout, wl.row_len).astype(np.float32)
    dead = np.flatnonzero(adv == 0)
    assert 0 < len(dead) < T
    N = int(wl.mask.sum())
    gs = np.float32(1.0 / N)
    rng = np.random.default_rng(14)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d_h = torch.full((T, Hd), 7.0, device=DEV)
    dW = torch.full((V, Hd), 7.0, device=DEV)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    terms = oterms = None
    w_tok = None
    ref_lp = None
    if with_terms:
        ref_lp = (-12.0 + rng.normal(0, 0.3, T)).astype(np.float32)
        w_tok = rng.choice([1.0, 0.5, 0.25], T).astype(np.float32)
        ent_t = torch.full((T,), -7.0, device=DEV)
        terms = dict(kl_kind=_lib.KL_K3, kl_coef=0.05, ref_logp=t(ref_lp), ent_coef=0.01, entropy_tok=ent_t,
                     w_tok=t(w_tok))
    _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), None, t(adv), t(wl.mask), wl.eps, float(gs), d_h, dW,
                                  loss, logp, acc, ws, terms=terms)
    res = _lib.grpo_finish_step(acc, loss, expected_N=N)
    assert res["status"] == 0 and res["n_valid"] == N and res["kernel_flags"] == 0
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 16383], rng.choice(dead, 3, replace=False),
                                     rng.choice(np.setdiff1d(np.arange(T), dead), 3, replace=False)]))
    hb = h[torch.from_numpy(rows).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
    wb = Wt.view(torch.int16).cpu().numpy().view(np.uint16)
    scale = (gs * w_tok[rows]).astype(np.float64) if with_terms else float(gs)
    if with_terms:
        oterms = dict(kl_kind=_lib.KL_K3, kl_coef=float(np.float32(0.05)), ref=ref_lp[rows].astype(np.float64),
                      ent_coef=float(np.float32(0.01)))
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target[rows], None, adv[rows], wl.mask[rows], wl.eps, scale=scale,
                            want_dw=False, terms=oterms)
    m = wl.mask[rows].astype(bool)
    gl, gp = H.to_f64(loss)[rows], H.to_f64(logp)[rows]
    assert np.all(np.abs(gp[m] - ref["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref["logp_tok"][m])))
    assert np.all(np.abs(gl - ref["loss_tok"]) <= 1e-5 * np.abs(ref["loss_tok"]) + 1e-6)
    if with_terms:
        ge = H.to_f64(ent_t)[rows]
        assert np.all(np.abs(ge[m] - ref["entropy"][m]) <= 1e-5 * np.maximum(1, ref["entropy"][m]))
    wf = OL.as_f64(wb)
    z = OL.as_f64(hb) @ wf.T
    awf = np.abs(wf)
    for k, tok in enumerate(rows):
        tt = None if not with_terms else dict(oterms, ref=float(ref_lp[tok]))
        sk = scale[k] if with_terms else scale
        dz = np.abs(OL.token_objective(z[k], int(wl.target[tok]), None, adv[tok], int(wl.mask[tok]), wl.eps, sk,
                                       terms=tt)[4])
        tol = 8e-3 * (dz @ awf) + 1e-12
        got = d_h[int(tok)].double().cpu().numpy()
        assert np.all(np.abs(got - ref["d_h"][k]) <= tol), int(tok)
    if not with_terms:
        assert torch.equal(d_h[torch.from_numpy(dead).to(DEV)], torch.zeros((len(dead), Hd), device=DEV))
    col = dW.double().sum(0)
    mag = dW.double().abs().sum(0)
    assert torch.all(col.abs() <= 2e-2 * mag + 1e-9)
    assert torch.isfinite(dW).all() and torch.isfinite(d_h).all()


def _random_case(k):
    """A seeded random LM-head case: sizes, dead fraction, clip stress, regularisers."""
    rng = np.random.default_rng(1000 + k)
    T = int(rng.integers(1, 700))
    V = int(rng.integers(1, 5000))
    Hd = int(rng.choice([64, 128, 192, 256]))
    dead_frac = float(rng.choice([0.0, 0.3, 0.7, 1.0]))
    # by k: no regulariser (the dead tokens skip the backward), KL k1, KL k3 with the entropy
    # bonus, no regulariser with weights
    kl = (0, _lib.KL_K1, _lib.KL_K3, 0)[k % 4]
    ent = 0.03 if k % 4 == 2 else 0.0
    weighted = k % 4 == 3 or bool(rng.integers(0, 2))
    return rng, T, V, Hd, dead_frac, kl, ent, weighted


@pytest.mark.parametrize("k", range(12))
def test_lmhead_random_cases(cta_group, k):
    # seeded random sizes (ragged tokens, vocabulary and K), a random share of tokens without a
    # gradient (zero advantage), masked tokens, random regularisers and weights, and half the
    # cases accumulating into a dW that already holds values; every output against the oracle
    rng, T, V, Hd, dead_frac, kl, ent, weighted = _random_case(k)
    adv = rng.choice([-1.5, -0.4, 0.6, 2.0], T).astype(np.float32)
    adv[rng.random(T) < dead_frac] = 0.0
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=2000 + k, valid_lo=0.15, adv=adv)
    N = max(int(mask.sum()), 1)
    gs = np.float32(1.0 / N)
    ref_lp = (old_logp + rng.normal(0, 0.3, T)).astype(np.float32)
    w_tok = rng.choice([1.0, 0.5, 0.125], T).astype(np.float32) if weighted else None
    accumulate = bool(k % 2)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d_h = torch.full((T, Hd), 7.0, device=DEV)
    dW0 = torch.randn((V, Hd), device=DEV) if accumulate else torch.full((V, Hd), 7.0, device=DEV)
    dW = dW0.clone()
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    ent_t = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
    terms = dict(kl_kind=kl, kl_coef=0.1, ref_logp=t(ref_lp) if kl else None, ent_coef=ent, entropy_tok=ent_t,
                 w_tok=t(w_tok))
    _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, float(gs), d_h, dW,
                                  loss, logp, acc, ws, dw_accumulate=accumulate, terms=terms)
    torch.cuda.synchronize()
    scale = (gs * w_tok).astype(np.float64) if weighted else float(gs)
    oterms = dict(kl_kind=kl, kl_coef=float(np.float32(0.1)), ref=ref_lp.astype(np.float64),
                  ent_coef=float(np.float32(ent)))
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=scale, terms=oterms)
    m = mask.astype(bool)
    gl, gp, ge = H.to_f64(loss), H.to_f64(logp), H.to_f64(ent_t)
    assert np.all(np.abs(gp[m] - ref["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref["logp_tok"][m])))
    assert np.all(np.abs(ge[m] - ref["entropy"][m]) <= 1e-5 * np.maximum(1, ref["entropy"][m]))
    assert np.all(gl[~m] == 0) and np.all(gp[~m] == 0) and np.all(ge[~m] == 0)
    assert np.all(np.abs(gl - ref["loss_tok"]) <= 1e-5 * np.abs(ref["loss_tok"]) + 1e-6)
    res = _lib.grpo_finish_step(acc, loss, expected_N=int(mask.sum()))
    assert res["status"] == 0 and res["kernel_flags"] == 0
    hf, wf = OL.as_f64(hb), OL.as_f64(wb)
    z = hf @ wf.T
    dz_abs = np.zeros_like(z)
    for i in range(T):
        if mask[i]:
            sk = scale[i] if weighted else scale
            dz_abs[i] = np.abs(OL.token_objective(z[i], int(wl.target[i]), old_logp[i], a_tok[i], 1, wl.eps, sk,
                                                  terms=dict(oterms, ref=float(ref_lp[i])))[4])
    gh = H.to_f64(d_h)
    bad = np.abs(gh - ref["d_h"]) > 8e-3 * (dz_abs @ np.abs(wf)) + 1e-12
    assert not bad.any(), (np.argwhere(bad)[:3], gh[bad][:3], ref["d_h"][bad][:3])
    want_w = ref["dW"] + (H.to_f64(dW0) if accumulate else 0.0)
    gw = H.to_f64(dW)
    tol_w = 8e-3 * (dz_abs.T @ np.abs(hf)) + 1e-12 + (2.0 ** -23) * np.abs(want_w)
    bad = np.abs(gw - want_w) > tol_w
    assert not bad.any(), (np.argwhere(bad)[:3], gw[bad][:3], want_w[bad][:3])
    # tokens without a gradient: an exact zero d_h row
    no_grad = ~np.any(dz_abs != 0, axis=1)
    assert np.all(gh[no_grad] == 0)


# ---- pass A over the valid tokens only (GRPO_LMHEAD_SKIP_MASKED) ------------------------------

@pytest.mark.parametrize("T, V, Hd, masked, with_terms", [(300, 3000, 128, 0.6, False), (513, 20000, 192, 0.3, True),
                                                          (256, 1024, 64, 0.0, False), (200, 2000, 64, 1.0, False),
                                                          (1, 777, 64, 0.0, True)])
def test_lmhead_skip_masked_gives_the_same_bits(cta_group, T, V, Hd, masked, with_terms):
    # pass A over the mask=1 tokens only (compact order, count on the device) against the call
    # that runs it over every token: every output the same bits, including with every token
    # masked or none, the regularisers, and a forward-only call
    rng = np.random.default_rng(int(T + V))
    wl, h, Wt, hb, wb, mask, a_tok, old_logp = _case(T, V, Hd, seed=101 + T)
    mask = (rng.random(T) >= masked).astype(np.uint8)
    a_tok = a_tok.copy()
    a_tok[: T // 4] = 0.0
    N = max(int(mask.sum()), 1)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    ref_lp = (old_logp + rng.normal(0, 0.3, T)).astype(np.float32)

    def call(skip, grads=True):
        o = dict(d_h=torch.full((T, Hd), 7.0, device=DEV) if grads else None,
                 dW=torch.full((V, Hd), 7.0, device=DEV) if grads else None,
                 loss=torch.full((T,), -7.0, device=DEV), logp=torch.full((T,), -7.0, device=DEV),
                 ent=torch.full((T,), -7.0, device=DEV), acc=_lib.new_step_acc(DEV))
        ws = torch.full((_lib.grpo_lmhead_workspace_size(T, V, Hd),), 0xFF, dtype=torch.uint8, device=DEV)
        terms = dict(kl_kind=_lib.KL_K3, kl_coef=0.1, ref_logp=t(ref_lp), ent_coef=0.02, entropy_tok=o["ent"]) \
            if with_terms else None
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old_logp), t(a_tok), t(mask), wl.eps, 1.0 / N,
                                      o["d_h"], o["dW"], o["loss"], o["logp"], o["acc"], ws, terms=terms,
                                      skip_masked=skip)
        o["res"] = _lib.grpo_finish_step(o["acc"], o["loss"], expected_N=int(mask.sum()))
        return o

    for grads in (True, False):
        a, b = call(False, grads), call(True, grads)
        for key in ("d_h", "dW", "loss", "logp", "ent"):
            if a[key] is not None:
                assert torch.equal(a[key], b[key]), key
        assert a["res"] == b["res"]
        assert b["res"]["status"] == 0 and b["res"]["kernel_flags"] == 0
    # and against the oracle
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_logp, a_tok, mask, wl.eps, scale=1.0 / N,
                            terms=dict(kl_kind=_lib.KL_K3, kl_coef=float(np.float32(0.1)),
                                       ref=ref_lp.astype(np.float64), ent_coef=float(np.float32(0.02)))
                            if with_terms else None)
    m = mask.astype(bool)
    gp = H.to_f64(b["logp"])
    assert np.all(np.abs(gp[m] - ref["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref["logp_tok"][m])))
    assert np.all(gp[~m] == 0) and np.all(H.to_f64(b["loss"])[~m] == 0)


def test_lmhead_another_model_shape_sampled_rows():
    # a Qwen2.5-7B-shaped head: H = 3584 (56 K blocks; d_h and dW over 14 column tiles) and
    # V = 152064 (594 vocabulary tiles, the last one whole); 640 tokens, a quarter of them
    # without a gradient. Sampled rows against the oracle row by row, dW by the vanishing
    # vocabulary sum.
    T, V, Hd = 640, 152064, 3584
    wl = W.make_workload("lmhead", seed=12, rows=8, tokens=T, V=V, H=Hd)
    h, Wt = W.make_lmhead_inputs(wl, DEV)
    rng = np.random.default_rng(13)
    adv = rng.choice([-1.0, 0.5, 1.5], T).astype(np.float32)
    adv[rng.random(T) < 0.25] = 0.0
    N = int(wl.mask.sum())
    d_h, dW, loss, logp, acc = _run(h, Wt, wl, wl.mask, adv, None, 1.0 / N)
    res = _lib.grpo_finish_step(acc, loss, expected_N=N)
    assert res["status"] == 0 and res["kernel_flags"] == 0
    rows = np.unique(np.concatenate([[0, 255, 256, 511, 639], rng.choice(T, 7, replace=False)]))
    hb = h[torch.from_numpy(rows).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
    wb = Wt.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = OL.lmhead_fwd_bwd(hb, wb, wl.target[rows], None, adv[rows], wl.mask[rows], wl.eps, scale=1.0 / N,
                            want_dw=False)
    H.assert_tokens_close(H.to_f64(loss)[rows], H.to_f64(logp)[rows], ref, adv[rows], wl.mask[rows])
    wf = OL.as_f64(wb)
    z = OL.as_f64(hb) @ wf.T
    awf = np.abs(wf)
    for k, tok in enumerate(rows):
        dz = np.abs(OL.token_objective(z[k], int(wl.target[tok]), None, adv[tok], 1, wl.eps, 1.0 / N)[4])
        got = d_h[int(tok)].double().cpu().numpy()
        assert np.all(np.abs(got - ref["d_h"][k]) <= 8e-3 * (dz @ awf) + 1e-12), int(tok)
        if adv[tok] == 0:
            assert np.all(got == 0)
    col = dW.double().sum(0)
    assert torch.all(col.abs() <= 2e-2 * dW.double().abs().sum(0) + 1e-9)
    assert torch.isfinite(dW).all() and torch.isfinite(d_h).all()
