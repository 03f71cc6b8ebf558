"""GPU parity: the library's loss forward/backward, advantage and step finish vs the oracle,
through the C ABI, on seeded inputs that span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

from oracle import advantage as OA
from oracle import loss as OL
from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import step as S
from rl_post_token_gb300 import workloads as W

from tests import _gpu_helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built(grpo_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return grpo_lib


def _run_direct(case, scale=1.0, want_grad=True, tok_src=None, old=True, logits=None):
    """One library call over all rows of a case."""
    T = case.logits.shape[0]
    lg = case.logits if logits is None else logits
    dl = torch.empty_like(lg) if want_grad else None
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd(lg, case.d_target, case.d_old if old else None, case.d_adv,
                                   case.d_mask, case.wl.eps, scale, dl, loss, logp, acc,
                                   tok_src=tok_src)
    torch.cuda.synchronize()
    return dl, loss, logp, acc


def _check_case(case, scale=1.0, old=True):
    dl, loss, logp, _ = _run_direct(case, scale, old=old)
    if not old:
        case_old, case.old = case.old, None
    ref = H.oracle_run(case, scale_per_token=np.full(case.logits.shape[0], scale))
    if not old:
        case.old = case_old
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, case.adv_tok, case.mask)
    amb = H.ambiguous_clip(ref["ratio"], case.wl.eps)
    alt = None
    if amb.any():
        alt = ref["dlogits"].copy()
        for t in np.nonzero(amb)[0]:
            z = OL.as_f64(case.logits_host[t])
            # the other clip decision: gradient on if it was off, off if it was on
            coef = 0.0 if not ref["clipped"][t] else case.adv_tok[t] * ref["ratio"][t] * scale
            alt[t] = coef * np.exp(OL.log_softmax_row(z))
            alt[t, case.target[t]] -= coef
    H.assert_dlogits_close(H.to_f64(dl), ref["dlogits"], case.wl.dtype, amb, alt,
                           target=ref["target"], coef=np.maximum(np.abs(ref["coef"]), np.abs(
                               case.adv_tok * ref["ratio"] * scale) * case.mask))
    return ref


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_workload_full(dtype):
    wl = W.make_workload("tiny", dtype=dtype)
    case = H.Case(wl)
    _check_case(case, scale=1.0 / 700)


@pytest.mark.parametrize("V", [1, 7, 1000, 4104, 8200, 65537])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_vocab(V, dtype):
    wl = W.make_workload("qwen_step", rows=4, len_lo=4, len_hi=7, V=V, dtype=dtype, seed=V)
    _check_case(H.Case(wl), scale=0.25)


def test_qwen_vocab_bf16():
    wl = W.make_workload("qwen_step", rows=4, len_lo=20, len_hi=40, seed=3)
    _check_case(H.Case(wl), scale=1.0 / 97)


def test_qwen_vocab_f32():
    wl = W.make_workload("qwen_step", rows=4, len_lo=3, len_hi=5, dtype="f32", seed=4)
    _check_case(H.Case(wl), scale=1.0)


def test_no_pi_old_ratio_one():
    wl = W.make_workload("qwen_step", rows=4, len_lo=8, len_hi=12, V=4104, seed=5)
    case = H.Case(wl)
    ref = _check_case(case, scale=0.5, old=False)
    assert np.all(ref["ratio"] == 1.0)


def test_stress_clip_binds():
    wl = W.make_workload("qwen_step", rows=4, len_lo=30, len_hi=60, V=8200, seed=6, old_sigma=0.5)
    adv = np.random.default_rng(6).choice([-1.5, -0.5, 0.5, 1.5], wl.T)
    case = H.Case(wl, adv_override=adv)
    ref = _check_case(case, scale=0.125)
    assert ref["clipped"].sum() > 10


def test_masked_and_zero_advantage_rows():
    wl = W.make_workload("tiny", rows=8, positions=40, valid_lo=0, V=2048, dtype="bf16", seed=8)
    case = H.Case(wl)
    case.adv_tok[:40] = 0.0  # a zero-variance group: the whole row has A = 0
    case.d_adv = torch.from_numpy(case.adv_tok).to(DEV)
    ref = _check_case(case, scale=0.01)
    dl, loss, logp, _ = _run_direct(case, 0.01)
    assert torch.all(dl[:40] == 0)
    assert np.all(ref["loss_tok"][wl.mask == 0] == 0)


def test_forward_only_matches_and_writes_no_grad():
    wl = W.make_workload("qwen_step", rows=4, len_lo=10, len_hi=20, V=8200, seed=9)
    case = H.Case(wl)
    _, loss, logp, acc = _run_direct(case, 1.0, want_grad=False)
    ref = H.oracle_run(case, want_grad=False)
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, case.adv_tok, case.mask)


def test_tok_src_permutation_and_padding_rows():
    wl = W.make_workload("qwen_step", rows=4, len_lo=4, len_hi=9, V=4104, seed=10)
    case = H.Case(wl)
    T = case.logits.shape[0]
    rng = np.random.default_rng(0)
    perm = rng.permutation(T)
    pads = rng.choice(T, 3)
    tok_src = np.concatenate([perm, -1 - pads]).astype(np.int64)
    lg = torch.cat([case.logits[torch.from_numpy(perm).to(DEV)], case.logits[torch.from_numpy(pads).to(DEV)]])
    dl, loss, logp, acc = _run_direct(case, 0.5, tok_src=torch.from_numpy(tok_src).to(DEV), logits=lg)
    ref = H.oracle_run(case, scale_per_token=np.full(T, 0.5))
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, case.adv_tok, case.mask)
    got = H.to_f64(dl)
    H.assert_dlogits_close(got[:T], ref["dlogits"][perm], "bf16", target=ref["target"][perm],
                           coef=ref["coef"][perm])
    assert np.all(got[T:] == 0)
    res = _lib.grpo_finish_step(acc, loss)
    assert res["n_tokens"] == T + 3 and res["n_valid"] == int(wl.mask.sum())


def test_empty_chunk_and_empty_step():
    acc = _lib.new_step_acc(DEV)
    e = torch.empty((0, 64), device=DEV)
    z = torch.empty(0, device=DEV)
    _lib.grpo_logprob_loss_fwd_bwd(e, torch.empty(0, dtype=torch.int32, device=DEV), None, z,
                                   torch.empty(0, dtype=torch.uint8, device=DEV), 0.2, 1.0, None, z, None, acc)
    res = _lib.grpo_finish_step(acc, z, expected_N=0)
    assert res["status"] == 0 and res["loss"] == 0.0 and res["n_valid"] == 0


def test_advantage_bit_exact_and_broadcast():
    rng = np.random.default_rng(12)
    for G, unbiased in [(4, True), (8, True), (2, False), (1, True)]:
        r = (rng.random(G * 16) < 0.3).astype(np.float32)
        r[:G] = 1.0  # an all-equal group
        r[G:2 * G] = rng.normal(size=G).astype(np.float32)
        d_r = torch.from_numpy(r).to(DEV)
        out = torch.empty_like(d_r)
        _lib.grpo_group_advantage(d_r, G, np.float32(1e-6), unbiased, out)
        want = OA.group_advantage(r, G, np.float32(1e-6), unbiased)
        assert np.array_equal(out.cpu().numpy(), want)
    # broadcast with a padding row (rollout -1)
    adv = torch.tensor([0.5, -1.0], device=DEV)
    rr = torch.tensor([0, 1, -1, 1], dtype=torch.int32, device=DEV)
    off = torch.tensor([0, 2, 3, 6, 8], dtype=torch.int64, device=DEV)
    tok = torch.full((8,), 9.0, device=DEV)
    rewards = torch.tensor([1.0, 0.0], device=DEV)
    _lib.grpo_group_advantage(rewards, 2, 1e-6, True, adv, rr, off, tok)
    a = adv.cpu().numpy()
    assert tok.cpu().numpy().tolist() == OA.broadcast_to_tokens(a, [0, 1, -1, 1], [2, 1, 3, 2]).tolist()


def test_chunked_equals_unchunked_bitwise():
    wl = W.make_workload("qwen_step", rows=8, len_lo=16, len_hi=40, V=8200, seed=13,
                         mini=4, micro=1)
    case = H.Case(wl)
    outs = []
    for micro in (1, 2, 4):
        cfg = dict(wl.plan, micro=micro)
        bp = S.plan_batch(cfg, wl.row_len, wl.row_valid)
        T = wl.T
        dl = torch.empty_like(case.logits)
        loss = torch.empty(T, device=DEV)
        logp = torch.empty(T, device=DEV)
        accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
        S.run_batch(bp, logits=case.logits, dlogits=dl, target=case.d_target, old_logp=case.d_old,
                    mask=case.d_mask, adv_tok=case.d_adv, loss_tok=loss, logp_tok=logp, accs=accs,
                    clip_eps=wl.eps)
        torch.cuda.synchronize()
        outs.append((dl.clone(), loss.clone(), S.read_results(accs, bp.n_steps)))
    for dl, loss, res in outs[1:]:
        assert torch.equal(dl.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(loss, outs[0][1])
        assert res == outs[0][2]
    # the step losses match the oracle's token mean over each mini-batch
    ref = H.oracle_run(case, want_grad=False)
    bp = S.plan_batch(dict(wl.plan, micro=1), wl.row_len, wl.row_valid)
    for s, (t0, t1) in enumerate(bp.step_tok_range):
        fin = OL.finish_step(ref["loss_tok"][t0:t1], wl.mask[t0:t1], ref["clipped"][t0:t1])
        got = outs[0][2][s]
        scale = max(abs(fin["loss"]), np.sum(np.abs(ref["loss_tok"][t0:t1])) / max(fin["n_valid"], 1))
        assert abs(got["loss"] - fin["loss"]) <= 1e-5 * scale
        assert got["n_valid"] == fin["n_valid"] == bp.plan["step_valid_tokens"][s]
        assert got["status"] == 0


def test_deferred_scaling_matches_direct_scale():
    wl = W.make_workload("qwen_step", rows=4, len_lo=10, len_hi=20, V=4104, seed=14)
    case = H.Case(wl)
    N = int(wl.mask.sum())
    dl, loss, logp, acc = _run_direct(case, 1.0)
    res = _lib.grpo_finish_step(acc, loss, expected_N=N, deferred=True, grad_bufs=[dl])
    assert res["status"] == 0 and res["n_valid"] == N
    ref = H.oracle_run(case, scale_per_token=np.full(wl.T, 1.0 / N))
    # two bf16 roundings (before and after the scale): allow twice the bf16 bar
    got = H.to_f64(dl)
    tol = H.dlogits_tol(ref["dlogits"], "bf16", ref["target"], ref["coef"], rel=2e-2)
    assert np.all(np.abs(got - ref["dlogits"]) <= tol)


def test_nonfinite_chunk_skips_step_and_zeroes_grads():
    wl = W.make_workload("qwen_step", rows=4, len_lo=6, len_hi=8, V=1000, seed=15)
    case = H.Case(wl)
    lg = case.logits.clone()
    lg[2, 17] = float("nan")   # a poisoned token row, planted in the host-side input
    dl, loss, logp, acc = _run_direct(case, 1.0, logits=lg)
    res = _lib.grpo_finish_step(acc, loss, grad_bufs=[dl])
    assert res["status"] == _lib.STEP_SKIPPED_NONFINITE and res["n_nonfinite"] >= 1
    assert torch.all(dl == 0)
    # the accumulator was reset: the next clean step is fine
    dl, loss, logp, acc2 = _run_direct(case, 1.0)
    assert _lib.grpo_finish_step(acc2, loss)["status"] == 0


def test_bad_target_counts_as_nonfinite():
    wl = W.make_workload("qwen_step", rows=4, len_lo=4, len_hi=5, V=1000, seed=16)
    case = H.Case(wl)
    case.d_target = case.d_target.clone()
    case.d_target[1] = 1000
    dl, loss, logp, acc = _run_direct(case, 1.0)
    assert _lib.grpo_finish_step(acc, loss)["n_nonfinite"] == 1


def test_expected_n_mismatch_reported():
    wl = W.make_workload("qwen_step", rows=4, len_lo=4, len_hi=5, V=1000, seed=17)
    case = H.Case(wl)
    dl, loss, logp, acc = _run_direct(case, 1.0)
    res = _lib.grpo_finish_step(acc, loss, expected_N=int(wl.mask.sum()) + 1, grad_bufs=[dl])
    assert res["status"] == _lib.ERR_N_MISMATCH
    assert torch.all(dl == 0)


def test_invalid_arguments_rejected():
    acc = _lib.new_step_acc(DEV)
    x = torch.zeros((2, 8), device=DEV)
    i = torch.zeros(2, dtype=torch.int32, device=DEV)
    m = torch.ones(2, dtype=torch.uint8, device=DEV)
    f = torch.zeros(2, device=DEV)
    with pytest.raises(_lib.GrpoError):
        _lib.grpo_logprob_loss_fwd_bwd(x, i, None, f, m, 0.2, 1.0, None, f, None, acc, V=9)
    with pytest.raises(_lib.GrpoError):
        _lib.grpo_logprob_loss_fwd_bwd(x, i, None, f, m, 0.2, 1.0, None, None, None, acc)


# ---- the shared-memory cluster kernel and its variants ---------------------------------------

VARIANTS = ["c2", "c3", "c4", "l2"]


@pytest.fixture
def variant(request, monkeypatch):
    monkeypatch.setenv("GRPO_ROWPASS", request.param)
    return request.param


@pytest.mark.parametrize("variant", VARIANTS, indirect=True)
@pytest.mark.parametrize("V,rows,positions", [(16384, 64, 12), (32776, 40, 10), (151936, 24, 12),
                                              (262144, 8, 10)])
def test_cluster_variants_many_rows_with_masks(variant, V, rows, positions):
    # many rows per cluster (refill pipeline, barrier phases), masked rows interleaved,
    # vocabularies whose last 16 KB chunk is ragged (32776) or that need 4-CTA clusters (262144)
    wl = W.make_workload("tiny", rows=rows, positions=positions, valid_lo=0, V=V, dtype="bf16",
                         seed=V % 997, std=3.0)
    _check_case(H.Case(wl), scale=1.0 / 333)


@pytest.mark.parametrize("variant", ["c2", "c3", "c4"], indirect=True)
def test_cluster_permutation_pad_rows_and_forward_only(variant):
    wl = W.make_workload("qwen_step", rows=8, len_lo=20, len_hi=40, V=16384, seed=21)
    case = H.Case(wl)
    T = case.logits.shape[0]
    rng = np.random.default_rng(1)
    perm = rng.permutation(T)
    pads = rng.choice(T, 5)
    tok_src = torch.from_numpy(np.concatenate([perm, -1 - pads]).astype(np.int64)).to(DEV)
    lg = torch.cat([case.logits[torch.from_numpy(perm).to(DEV)], case.logits[torch.from_numpy(pads).to(DEV)]])
    dl, loss, logp, acc = _run_direct(case, 0.5, tok_src=tok_src, logits=lg)
    ref = H.oracle_run(case, scale_per_token=np.full(T, 0.5))
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, case.adv_tok, case.mask)
    got = H.to_f64(dl)
    H.assert_dlogits_close(got[:T], ref["dlogits"][perm], "bf16", target=ref["target"][perm],
                           coef=ref["coef"][perm])
    assert np.all(got[T:] == 0)
    _, loss2, logp2, _ = _run_direct(case, 0.5, want_grad=False, tok_src=tok_src, logits=lg)
    assert torch.equal(loss2, loss) and torch.equal(logp2, logp)


@pytest.mark.parametrize("variant", ["c2", "c3", "c4"], indirect=True)
def test_cluster_nonfinite_row(variant):
    wl = W.make_workload("qwen_step", rows=4, len_lo=30, len_hi=40, V=16384, seed=22)
    case = H.Case(wl)
    lg = case.logits.clone()
    lg[7, 12000] = float("inf")
    lg[19, 3] = float("nan")
    dl, loss, logp, acc = _run_direct(case, 1.0, logits=lg)
    res = _lib.grpo_finish_step(acc, loss, grad_bufs=[dl])
    assert res["status"] == _lib.STEP_SKIPPED_NONFINITE and res["n_nonfinite"] == 2
    assert res["kernel_flags"] == 0
    assert torch.all(dl == 0)


@pytest.mark.parametrize("variant", ["c2", "c3", "c4"], indirect=True)
def test_cluster_chunked_equals_unchunked_bitwise(variant):
    wl = W.make_workload("qwen_step", rows=8, len_lo=16, len_hi=40, V=32776, seed=23, mini=4, micro=1)
    case = H.Case(wl)
    outs = []
    for micro in (1, 4):
        bp = S.plan_batch(dict(wl.plan, micro=micro), wl.row_len, wl.row_valid)
        dl = torch.empty_like(case.logits)
        loss = torch.empty(wl.T, device=DEV)
        logp = torch.empty(wl.T, device=DEV)
        accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
        S.run_batch(bp, logits=case.logits, dlogits=dl, target=case.d_target, old_logp=case.d_old,
                    mask=case.d_mask, adv_tok=case.d_adv, loss_tok=loss, logp_tok=logp, accs=accs,
                    clip_eps=wl.eps)
        torch.cuda.synchronize()
        outs.append((dl.view(torch.int16).clone(), loss.clone(), S.read_results(accs, bp.n_steps)))
    for o in outs[1:]:
        assert torch.equal(outs[0][0], o[0]) and torch.equal(outs[0][1], o[1])
        assert outs[0][2] == o[2]


@pytest.mark.parametrize("V", [16384, 32776, 151936])
def test_ring_slots_equal_fixed_buffer_bitwise(V, monkeypatch):
    # The shared-memory ring only changes where a chunk waits and when it is copied, never
    # the arithmetic: the fixed staging buffer (0), a ring with one spare slot or less (6) and
    # the default ring must give the same bits. 16384: a whole row per chunk; 32776: the two
    # CTAs of a cluster hold different chunk counts; 151936: the product vocabulary.
    monkeypatch.setenv("GRPO_ROWPASS", "c2")
    wl = W.make_workload("tiny", rows=12, positions=20, valid_lo=0, V=V, dtype="bf16", seed=V % 389, std=2.0)
    case = H.Case(wl)
    T = case.logits.shape[0]
    rng = np.random.default_rng(3)
    perm = rng.permutation(T)
    pads = rng.choice(T, 9)
    src = np.concatenate([perm, -1 - pads]).astype(np.int64)
    rng.shuffle(src)
    tok_src = torch.from_numpy(src).to(DEV)
    lg = case.logits[torch.from_numpy(np.where(src >= 0, src, -1 - src)).to(DEV)]
    outs = {}
    for slots in ("0", "6", None):
        if slots is None:
            monkeypatch.delenv("GRPO_ROWPASS_SLOTS", raising=False)
        else:
            monkeypatch.setenv("GRPO_ROWPASS_SLOTS", slots)
        dl, loss, logp, acc = _run_direct(case, 1.0 / 97, tok_src=tok_src, logits=lg)
        res = _lib.grpo_finish_step(acc, loss, expected_N=int(case.mask.sum()))
        outs[slots] = (dl.view(torch.int16).clone(), loss.clone(), logp.clone(), res)
        # forward only (slots released as soon as pass 1 is done with them): same per-token bits
        _, loss_f, logp_f, acc_f = _run_direct(case, 1.0 / 97, want_grad=False, tok_src=tok_src, logits=lg)
        res_f = _lib.grpo_finish_step(acc_f, loss_f, expected_N=int(case.mask.sum()))
        assert torch.equal(loss_f, loss) and torch.equal(logp_f, logp), slots
        assert res_f == res, slots
    for k in ("6", None):
        assert torch.equal(outs[k][0], outs["0"][0]), k
        assert torch.equal(outs[k][1], outs["0"][1]) and torch.equal(outs[k][2], outs["0"][2]), k
        assert outs[k][3] == outs["0"][3], k
    assert outs[None][3]["status"] == 0


@pytest.mark.parametrize("dtype,V,rows", [("bf16", 151936, 16), ("bf16", 32776, 32), ("f32", 32776, 32),
                                          ("bf16", 262144, 8)])
def test_forward_only_streaming_kernel_equals_general_bitwise(dtype, V, rows, monkeypatch):
    # Forward-only calls run the streaming kernel: slots released during pass 1, partials sent
    # to CTA 0 and combined one row late by a rotating warp. It must give the bits of the
    # general cluster kernel called forward only (GRPO_ROWPASS_FWD=0) at every ring size
    # (0 = two slots, the fewest), with masked and padding rows in a shuffled order, pi_old
    # given, more read rows per cluster than exchange buffers, and a valid token whose target
    # is out of range (its loss is NaN and it counts as non-finite). 262144: the 4-CTA
    # instance a bf16 row too long for two CTAs takes.
    wl = W.make_workload("tiny", rows=rows, positions=64, valid_lo=0, V=V, dtype=dtype, seed=V % 541 + rows,
                         std=2.0)
    case = H.Case(wl)
    T = case.logits.shape[0]
    rng = np.random.default_rng(7)
    perm = rng.permutation(T)
    pads = rng.choice(T, 11)
    src = np.concatenate([perm, -1 - pads]).astype(np.int64)
    rng.shuffle(src)
    tok_src = torch.from_numpy(src).to(DEV)
    lg = case.logits[torch.from_numpy(np.where(src >= 0, src, -1 - src)).to(DEV)]
    bad = int(np.nonzero(case.mask)[0][5])
    tgt = case.d_target.clone()
    tgt[bad] = V

    def run():
        loss = torch.full((T,), -7.0, device=DEV)
        logp = torch.full((T,), -7.0, device=DEV)
        acc = _lib.new_step_acc(DEV)
        _lib.grpo_logprob_loss_fwd_bwd(lg, tgt, case.d_old, case.d_adv, case.d_mask, wl.eps, 1.0 / 89, None,
                                       loss, logp, acc, tok_src=tok_src)
        torch.cuda.synchronize()
        return loss.view(torch.int32).clone(), logp.view(torch.int32).clone(), acc.clone()

    monkeypatch.setenv("GRPO_ROWPASS_FWD", "0")
    want = run()
    monkeypatch.delenv("GRPO_ROWPASS_FWD")
    for slots in ("0", "3", None):
        if slots is None:
            monkeypatch.delenv("GRPO_ROWPASS_SLOTS", raising=False)
        else:
            monkeypatch.setenv("GRPO_ROWPASS_SLOTS", slots)
        got = run()
        for g, w, what in zip(got, want, ("loss", "logp", "acc")):
            assert torch.equal(g, w), (slots, what)
    res = _lib.grpo_finish_step(want[2].clone(), want[0].view(torch.float32))
    assert res["status"] == _lib.STEP_SKIPPED_NONFINITE
    assert res["n_nonfinite"] == 1 and res["kernel_flags"] == 0
    assert res["n_tokens"] == T + 11 and res["n_valid"] == int(case.mask.sum())
    # and against the oracle (outputs are indexed by input token), every token but the one
    # with the bad target
    got_loss = want[0].view(torch.float32).cpu().numpy().astype(np.float64)
    got_logp = want[1].view(torch.float32).cpu().numpy().astype(np.float64)
    ref = H.oracle_run(case, want_grad=False)
    m = case.mask.copy()
    m[bad] = 0
    got_loss[bad] = got_logp[bad] = 0.0
    ref["loss_tok"][bad] = ref["logp_tok"][bad] = 0.0
    H.assert_tokens_close(got_loss, got_logp, ref, case.adv_tok, m)


@pytest.mark.parametrize("V", [16384, 32776, 151936])
def test_f32_cluster_rows_against_oracle(V, monkeypatch):
    # float32 logits through the 4-CTA cluster kernel: masked and padding rows, the four
    # slices of unequal length at V = 32776, forward-only bits equal to the full pass, and the
    # fixed staging buffer giving the same bits as the ring
    wl = W.make_workload("tiny", rows=8, positions=10, valid_lo=0, V=V, dtype="f32", seed=V % 211, std=2.0)
    case = H.Case(wl)
    T = case.logits.shape[0]
    rng = np.random.default_rng(4)
    perm = rng.permutation(T)
    pads = rng.choice(T, 4)
    src = np.concatenate([perm, -1 - pads]).astype(np.int64)
    tok_src = torch.from_numpy(src).to(DEV)
    lg = case.logits[torch.from_numpy(np.where(src >= 0, src, -1 - src)).to(DEV)]
    dl, loss, logp, acc = _run_direct(case, 1.0 / 53, tok_src=tok_src, logits=lg)
    ref = H.oracle_run(case, scale_per_token=np.full(T, 1.0 / 53))
    H.assert_tokens_close(H.to_f64(loss), H.to_f64(logp), ref, case.adv_tok, case.mask)
    got = H.to_f64(dl)
    H.assert_dlogits_close(got[:T], ref["dlogits"][perm], "f32", target=ref["target"][perm],
                           coef=ref["coef"][perm])
    assert np.all(got[T:] == 0)
    _, loss_f, logp_f, _ = _run_direct(case, 1.0 / 53, want_grad=False, tok_src=tok_src, logits=lg)
    assert torch.equal(loss_f, loss) and torch.equal(logp_f, logp)
    monkeypatch.setenv("GRPO_ROWPASS_SLOTS", "0")
    dl0, loss0, _, _ = _run_direct(case, 1.0 / 53, tok_src=tok_src, logits=lg)
    assert torch.equal(dl0, dl) and torch.equal(loss0, loss)


@pytest.mark.parametrize("kl_kind,ent", [(2, 0.0), (0, 0.02)])
def test_f32_cluster_terms(kl_kind, ent):
    wl = W.make_workload("tiny", rows=4, positions=12, valid_lo=0, V=32776, dtype="f32", seed=60 + kl_kind, std=2.0)
    case = H.Case(wl)
    T = wl.T
    ref = (case.old + np.random.default_rng(3).normal(0, 0.3, T)).astype(np.float32)
    scale = 1.0 / 41
    dl = torch.empty_like(case.logits)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    ent_t = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd(case.logits, case.d_target, case.d_old, case.d_adv, case.d_mask, wl.eps,
                                   scale, dl, loss, logp, acc,
                                   terms=dict(kl_kind=kl_kind, kl_coef=0.1, ref_logp=torch.from_numpy(ref).to(DEV),
                                              ent_coef=ent, entropy_tok=ent_t))
    torch.cuda.synchronize()
    out = OL.loss_fwd_bwd(case.logits_host, wl.target, case.old, case.adv_tok, wl.mask, wl.eps, scale, True,
                          dict(kl_kind=kl_kind, kl_coef=float(np.float32(0.1)), ref=ref.astype(np.float64),
                               ent_coef=float(np.float32(ent))))
    m = wl.mask.astype(bool)
    assert np.all(np.abs(H.to_f64(ent_t)[m] - out["entropy"][m]) <= 1e-5 * np.maximum(1, out["entropy"][m]))
    assert np.all(np.abs(H.to_f64(loss) - out["loss_tok"]) <= 1e-5 * np.abs(out["loss_tok"]) + 1e-6)
    got, refd = H.to_f64(dl), out["dlogits"]
    amb = H.ambiguous_clip(out["ratio"], wl.eps)
    probs = H.row_probs(case.logits_host) if ent else None
    bad = np.abs(got - refd) > H.dlogits_tol(refd, "f32", probs=probs)
    bad[amb] = False
    assert not bad.any(), np.argwhere(bad)[:3]


def test_cluster_long_masked_runs(monkeypatch):
    # Read rows only in three short windows, separated by masked runs several grid strides
    # long: the producer's look-ahead skips many rows at a time and a third of the clusters
    # read no row at all; every row still gets its loss and its (zero or full) dlogits row.
    monkeypatch.setenv("GRPO_ROWPASS", "c2")
    wl = W.make_workload("tiny", rows=20, positions=30, valid_lo=0, V=16384, dtype="bf16", seed=41, std=2.0)
    case = H.Case(wl)
    T = case.logits.shape[0]
    assert T == 600
    m = np.zeros(T, np.uint8)
    m[0:5] = 1
    m[310:330] = 1
    m[590:600] = 1
    case.mask = m
    case.d_mask = torch.from_numpy(m).to(DEV)
    _check_case(case, scale=1.0 / 35)


@pytest.mark.parametrize("variant", ["c2", "l2"], indirect=True)
def test_dynamic_bins_equal_fixed_chunks_bitwise(variant):
    # one mini-batch planned as fixed chunks and as token-budget bins (rows reordered, chunk
    # boundaries moved): every token's loss, log-prob and dlogits row is bit-identical, and so
    # are the step results
    wl = W.make_workload("qwen_step", rows=8, len_lo=8, len_hi=60, V=32776, seed=31, mini=8, micro=2)
    case = H.Case(wl)
    outs = []
    for cfg in (dict(wl.plan), dict(wl.plan, dynamic=1, max_token_len=128, workload=1, balance_ends=1)):
        bp = S.plan_batch(cfg, wl.row_len, wl.row_valid)
        src = np.arange(wl.T) if bp.tok_src is None else bp.tok_src
        lg = case.logits[torch.from_numpy(src).to(DEV)]  # exec order, as a model would emit it
        dl = torch.empty_like(lg)
        loss = torch.empty(wl.T, device=DEV)
        logp = torch.empty(wl.T, device=DEV)
        accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
        S.run_batch(bp, logits=lg, dlogits=dl, target=case.d_target, old_logp=case.d_old, mask=case.d_mask,
                    adv_tok=case.d_adv, loss_tok=loss, logp_tok=logp, accs=accs, clip_eps=wl.eps,
                    tok_src=None if bp.tok_src is None else torch.from_numpy(bp.tok_src).to(DEV))
        torch.cuda.synchronize()
        back = torch.empty_like(dl)
        back[torch.from_numpy(src).to(DEV)] = dl  # dlogits rows back to input order
        outs.append((bp.plan["n_chunks"], back.view(torch.int16), loss, logp, S.read_results(accs, bp.n_steps)))
    assert outs[0][0] != outs[1][0]  # the two schedules really differ
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][2], outs[1][2]) and torch.equal(outs[0][3], outs[1][3])
    assert outs[0][4] == outs[1][4]


# ---- regularisers: KL to the reference policy and the entropy bonus ----------------------------

@pytest.mark.parametrize("variant", ["c2", "c4", "l2"], indirect=True)
@pytest.mark.parametrize("kl_kind,ent", [(1, 0.0), (2, 0.0), (0, 0.02), (2, 0.05)])
def test_kl_and_entropy_terms(variant, kl_kind, ent):
    wl = W.make_workload("tiny", rows=8, positions=24, valid_lo=0, V=32776, dtype="bf16", seed=50 + kl_kind,
                         std=3.0)
    case = H.Case(wl)
    T = wl.T
    ref = (case.old + np.random.default_rng(3).normal(0, 0.3, T)).astype(np.float32)
    scale = 1.0 / 97
    dl = torch.empty_like(case.logits)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    ent_t = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    terms = dict(kl_kind=kl_kind, kl_coef=0.1, ref_logp=torch.from_numpy(ref).to(DEV), ent_coef=ent,
                 entropy_tok=ent_t)
    _lib.grpo_logprob_loss_fwd_bwd(case.logits, case.d_target, case.d_old, case.d_adv, case.d_mask, wl.eps,
                                   scale, dl, loss, logp, acc, terms=terms)
    torch.cuda.synchronize()
    oterms = dict(kl_kind=kl_kind, kl_coef=float(np.float32(0.1)), ref=ref.astype(np.float64),
                  ent_coef=float(np.float32(ent)))
    ref_out = OL.loss_fwd_bwd(case.logits_host, wl.target, case.old, case.adv_tok, wl.mask, wl.eps,
                              scale, True, oterms)
    m = wl.mask.astype(bool)
    gl, gp, ge = H.to_f64(loss), H.to_f64(logp), H.to_f64(ent_t)
    assert np.all(np.abs(gp[m] - ref_out["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref_out["logp_tok"][m])))
    assert np.all(np.abs(ge[m] - ref_out["entropy"][m]) <= 1e-5 * np.maximum(1, ref_out["entropy"][m]))
    assert np.all(ge[~m] == 0) and np.all(gl[~m] == 0)
    assert np.all(np.abs(gl - ref_out["loss_tok"]) <= 1e-5 * np.abs(ref_out["loss_tok"]) + 1e-6)
    # dlogits: every element relative to its own value (plus the entropy term's float32
    # difference when the bonus is on), except the ambiguous-clip rows of the smaller tests
    amb = H.ambiguous_clip(ref_out["ratio"], wl.eps)
    got = H.to_f64(dl)
    refd = ref_out["dlogits"]
    probs = H.row_probs(case.logits_host) if ent else None
    bad = np.abs(got - refd) > H.dlogits_tol(refd, "bf16", probs=probs)
    bad[amb] = False
    assert not bad.any(), np.argwhere(bad)[:3]
    res = _lib.grpo_finish_step(acc, loss)
    assert res["status"] == 0 and res["n_valid"] == int(wl.mask.sum())


@pytest.mark.parametrize("kind", ["fixed", "dynamic"])
def test_driver_loop_terms_equal_direct_calls_bitwise(kind):
    # KL (k3) and the entropy bonus through the driver loop: a step's chunks alternate over two
    # streams, and for token-budget bins the order is permuted (the terms' per-token arrays are
    # then read through the token index). Every token's loss, log-prob, entropy and dlogits row
    # equals one direct call per optimizer step over its tokens in input order, bit for bit.
    if kind == "fixed":
        wl = W.make_workload("tiny", rows=8, positions=24, valid_lo=0, V=32776, dtype="bf16", seed=93, std=2.0,
                             mini=4, micro=2)
    else:
        wl = W.make_workload("dynamic", rows=16, len_hi=64, median=20, max_token_len=96, V=32776, seed=94)
    case = H.Case(wl)
    T = wl.T
    ref = torch.from_numpy((case.old + np.random.default_rng(5).normal(0, 0.3, T)).astype(np.float32)).to(DEV)
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    assert bp.n_steps == (2 if kind == "fixed" else 1) and bp.plan["n_chunks"] >= 3
    assert (bp.tok_src is None) == (kind == "fixed")
    src = np.arange(bp.exec_tokens) if bp.tok_src is None else bp.tok_src
    assert np.all(src >= 0)
    lg = case.logits[torch.from_numpy(src).to(DEV)]  # exec order
    dl = torch.empty_like(lg)
    loss, logp, ent = (torch.full((T,), -7.0, device=DEV) for _ in range(3))
    accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
    terms = dict(kl_kind=_lib.KL_K3, kl_coef=0.1, ref_logp=ref, ent_coef=0.02, entropy_tok=ent)
    S.run_batch(bp, logits=lg, dlogits=dl, target=case.d_target, old_logp=case.d_old, mask=case.d_mask,
                adv_tok=case.d_adv, loss_tok=loss, logp_tok=logp, accs=accs, clip_eps=wl.eps,
                tok_src=None if bp.tok_src is None else torch.from_numpy(bp.tok_src).to(DEV),
                side_stream=torch.cuda.Stream(), terms=terms)
    torch.cuda.synchronize()
    res = S.read_results(accs, bp.n_steps)
    back = torch.empty_like(dl)
    back[torch.from_numpy(src).to(DEV)] = dl  # dlogits rows back to input order
    for k in range(bp.n_steps):
        t0, t1 = bp.step_tok_range[k]
        N = int(bp.plan["step_valid_tokens"][k])
        dl_k = torch.empty_like(case.logits[t0:t1])
        loss_k, logp_k, ent_k = (torch.full((t1 - t0,), -7.0, device=DEV) for _ in range(3))
        acc_k = _lib.new_step_acc(DEV)
        _lib.grpo_logprob_loss_fwd_bwd(case.logits[t0:t1], case.d_target[t0:t1], case.d_old[t0:t1],
                                       case.d_adv[t0:t1], case.d_mask[t0:t1], wl.eps, 1.0 / max(N, 1), dl_k,
                                       loss_k, logp_k, acc_k,
                                       terms=dict(terms, ref_logp=ref[t0:t1], entropy_tok=ent_k))
        torch.cuda.synchronize()
        for got, want in ((loss[t0:t1], loss_k), (logp[t0:t1], logp_k), (ent[t0:t1], ent_k)):
            assert torch.equal(got.view(torch.int32), want.view(torch.int32)), k
        assert torch.equal(back[t0:t1].view(torch.int16), dl_k.view(torch.int16)), k
        direct = _lib.grpo_finish_step(acc_k, loss_k, expected_N=N)
        for key in ("loss", "n_valid", "n_clipped", "n_nonfinite", "n_tokens", "status"):
            assert res[k][key] == direct[key], (k, key)


@pytest.mark.parametrize("variant", ["c2", "c4", "l2"], indirect=True)
def test_entropy_with_masked_vocabulary(variant):
    # A tenth of every row's vocabulary is -inf (a masked vocabulary; never the target): those
    # elements carry no mass, add nothing to sum p z (p log p -> 0), and get a zero gradient.
    wl = W.make_workload("tiny", rows=8, positions=16, valid_lo=0, V=32776, dtype="bf16", seed=61, std=2.0)
    case = H.Case(wl)
    T, V = wl.T, wl.V
    rng = np.random.default_rng(5)
    off = rng.random((T, V)) < 0.1
    off[np.arange(T), wl.target] = False
    lg = case.logits.clone()
    lg[torch.from_numpy(off).to(DEV)] = float("-inf")
    host = W.logits_to_host(lg)
    scale = 1.0 / 61
    dl = torch.empty_like(lg)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    ent_t = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd(lg, case.d_target, case.d_old, case.d_adv, case.d_mask, wl.eps, scale, dl,
                                   loss, logp, acc, terms=dict(ent_coef=0.03, entropy_tok=ent_t))
    torch.cuda.synchronize()
    ref_out = OL.loss_fwd_bwd(host, wl.target, case.old, case.adv_tok, wl.mask, wl.eps, scale, True,
                              dict(kl_kind=0, kl_coef=0.0, ref=None, ent_coef=float(np.float32(0.03))))
    m = wl.mask.astype(bool)
    ge, gp = H.to_f64(ent_t), H.to_f64(logp)
    assert np.all(np.isfinite(ge)) and np.all(np.isfinite(gp))
    assert np.all(np.abs(ge[m] - ref_out["entropy"][m]) <= 1e-5 * np.maximum(1, ref_out["entropy"][m]))
    assert np.all(np.abs(gp[m] - ref_out["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref_out["logp_tok"][m])))
    got = H.to_f64(dl)
    assert np.all(np.isfinite(got)) and np.all(got[off] == 0)
    refd = ref_out["dlogits"]
    amb = H.ambiguous_clip(ref_out["ratio"], wl.eps)
    bad = np.abs(got - refd) > H.dlogits_tol(refd, "bf16", probs=H.row_probs(host))
    bad[amb] = False
    assert not bad.any(), np.argwhere(bad)[:3]
    res = _lib.grpo_finish_step(acc, loss)
    assert res["status"] == 0 and res["n_nonfinite"] == 0


@pytest.mark.parametrize("variant", ["c2", "c4", "l2"], indirect=True)
def test_plain_and_forward_only_with_masked_vocabulary(variant):
    # -inf logits in the plain instance and the forward-only pass: a tenth of every row at
    # random, every row's first element (the lazy shift's starting point), and a run of 4096
    # (whole per-thread blocks of -inf), never the target. They carry no mass, their dlogits
    # are exactly 0, every output is finite, and the forward-only pass gives the full pass's bits.
    wl = W.make_workload("tiny", rows=8, positions=16, valid_lo=0, V=32776, dtype="bf16", seed=62, std=2.0)
    case = H.Case(wl)
    T, V = wl.T, wl.V
    rng = np.random.default_rng(6)
    off = rng.random((T, V)) < 0.1
    off[:, 0] = True
    off[:, 8192:8192 + 4096] = True
    off[np.arange(T), wl.target] = False
    lg = case.logits.clone()
    lg[torch.from_numpy(off).to(DEV)] = float("-inf")
    host = W.logits_to_host(lg)
    scale = 1.0 / 59
    dl, loss, logp, acc = _run_direct(case, scale, logits=lg)
    ref_out = OL.loss_fwd_bwd(host, wl.target, case.old, case.adv_tok, wl.mask, wl.eps, scale, True)
    m = wl.mask.astype(bool)
    gp, gl = H.to_f64(logp), H.to_f64(loss)
    assert np.all(np.isfinite(gp)) and np.all(np.isfinite(gl))
    assert np.all(np.abs(gp[m] - ref_out["logp_tok"][m]) <= 1e-5 * np.maximum(1, np.abs(ref_out["logp_tok"][m])))
    got = H.to_f64(dl)
    assert np.all(np.isfinite(got)) and np.all(got[off] == 0)
    refd = ref_out["dlogits"]
    bad = np.abs(got - refd) > H.dlogits_tol(refd, "bf16")
    bad[H.ambiguous_clip(ref_out["ratio"], wl.eps)] = False
    assert not bad.any(), np.argwhere(bad)[:3]
    res = _lib.grpo_finish_step(acc, loss)
    assert res["status"] == 0 and res["n_nonfinite"] == 0
    _, loss_f, logp_f, _ = _run_direct(case, scale, want_grad=False, logits=lg)
    assert torch.equal(loss_f, loss) and torch.equal(logp_f, logp)


def test_terms_reject_bad_arguments():
    acc = _lib.new_step_acc(DEV)
    x = torch.zeros((2, 8), device=DEV)
    i = torch.zeros(2, dtype=torch.int32, device=DEV)
    mk = torch.ones(2, dtype=torch.uint8, device=DEV)
    f = torch.zeros(2, device=DEV)
    with pytest.raises(_lib.GrpoError):
        _lib.grpo_logprob_loss_fwd_bwd(x, i, None, f, mk, 0.2, 1.0, None, f, None, acc, terms=dict(kl_kind=7))
    with pytest.raises(_lib.GrpoError):
        _lib.grpo_logprob_loss_fwd_bwd(x, i, None, f, mk, 0.2, 1.0, None, f, None, acc, terms=dict(kl_kind=1))


def test_concurrent_host_threads_bitwise():
    # two host threads, two streams, two vocabularies (two shared-memory sizes of the cluster
    # kernel), launching at once: every result equals the single-threaded one bit for bit
    import threading

    cases = []
    for V, seed in ((16384, 91), (151936, 92)):
        wl = W.make_workload("tiny", rows=4, positions=12, valid_lo=0, V=V, dtype="bf16", seed=seed, std=2.0)
        cases.append(H.Case(wl))

    def run(case, stream, n):
        outs = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                T = case.logits.shape[0]
                dl = torch.empty_like(case.logits)
                loss = torch.empty(T, device=DEV)
                acc = _lib.new_step_acc(DEV)
                _lib.grpo_logprob_loss_fwd_bwd(case.logits, case.d_target, case.d_old, case.d_adv, case.d_mask,
                                               case.wl.eps, 1.0 / 41, dl, loss, None, acc, stream=stream)
                outs.append((dl, loss))
        stream.synchronize()
        return outs

    ref = [run(c, torch.cuda.Stream(), 1)[0] for c in cases]
    got = [None, None]
    errs = []

    def worker(i):
        try:
            got[i] = run(cases[i], torch.cuda.Stream(), 12)
        except Exception as e:  # surfaced below
            errs.append(e)

    th = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errs, errs
    for i in range(2):
        for dl, loss in got[i]:
            assert torch.equal(dl.view(torch.int16), ref[i][0].view(torch.int16))
            assert torch.equal(loss, ref[i][1])


@pytest.mark.parametrize("deferred", [False, True])
def test_two_stream_chunks_bitwise(deferred):
    # a step's chunks rotating over two or three streams (overlapping at their ends), and each
    # step's finish on a stream of its own while the next step's chunks run, give the same bits
    # as one stream: dlogits (in deferred mode scaled by the finish), per-token losses and the
    # step results
    wl = W.make_workload("qwen_step", rows=8, len_lo=16, len_hi=40, V=32776, seed=27, mini=4, micro=1)
    case = H.Case(wl)
    side, fin = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for ss, fs in ((None, None), (side, None), ([side, torch.cuda.Stream()], None), (side, fin), (None, fin)):
        bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid)
        dl = torch.empty_like(case.logits)
        loss = torch.empty(wl.T, device=DEV)
        accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
        S.run_batch(bp, logits=case.logits, dlogits=dl, target=case.d_target, old_logp=case.d_old,
                    mask=case.d_mask, adv_tok=case.d_adv, loss_tok=loss, logp_tok=None, accs=accs,
                    clip_eps=wl.eps, side_stream=ss, finish_stream=fs, deferred=deferred)
        torch.cuda.synchronize()
        outs.append((dl.view(torch.int16).clone(), loss.clone(), S.read_results(accs, bp.n_steps)))
    for o in outs[1:]:
        assert torch.equal(outs[0][0], o[0]) and torch.equal(outs[0][1], o[1])
        assert outs[0][2] == o[2]


def test_bounded_wait_gives_up_and_the_step_reports_it():
    # The bounded waits every pipelined kernel relies on: a wait that nothing completes gives
    # up at its limit (about a second) instead of hanging, raises the wait-timeout flag, the
    # step finish reports ERR_KERNEL and zeroes the gradients, and the context stays usable.
    import time
    wl = W.make_workload("tiny", rows=4, positions=8, valid_lo=0, V=16384, dtype="bf16", seed=71, std=2.0)
    case = H.Case(wl)
    dl, loss, logp, acc = _run_direct(case, 0.5)
    t0 = time.perf_counter()
    _lib.grpo_selftest_wait_timeout(acc)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    res = _lib.grpo_finish_step(acc, loss, grad_bufs=[dl])
    assert res["status"] == _lib.ERR_KERNEL and res["kernel_flags"] == 1
    assert torch.all(dl == 0)
    # the flag was consumed by the finish, and the device still runs the path normally
    dl2, loss2, logp2, acc2 = _run_direct(case, 0.5)
    res2 = _lib.grpo_finish_step(acc2, loss2, grad_bufs=[dl2])
    assert res2["status"] == 0 and res2["kernel_flags"] == 0
    assert torch.equal(loss2, loss) and torch.equal(logp2, logp)


@pytest.mark.parametrize("dtype,V,block,pinned,permuted,two_streams", [
    ("bf16", 32776, 37, True, True, True), ("bf16", 151936, 64, True, False, True),
    ("f32", 16384, 50, False, True, False), ("bf16", 32776, 1000, True, True, True)])
def test_host_logits_streaming_equals_device_call(dtype, V, block, pinned, permuted, two_streams):
    # Logits in host memory, streamed through a two-block device staging buffer (copies on a
    # second stream, each block's row pass waiting only for its own copy): the bits of the
    # device call on the same rows. Ragged blocks, a permuted order with padding rows or the
    # identity order, pi_old, the KL and entropy terms; pageable host memory and a single
    # stream too; a block larger than the call.
    wl = W.make_workload("tiny", rows=12, positions=20, valid_lo=0, V=V, dtype=dtype, seed=V % 331 + block, std=2.0)
    case = H.Case(wl)
    T = case.logits.shape[0]
    rng = np.random.default_rng(9)
    tok_src, lg = None, case.logits
    if permuted:
        src = np.concatenate([rng.permutation(T), -1 - rng.choice(T, 5)]).astype(np.int64)
        rng.shuffle(src)
        tok_src = torch.from_numpy(src).to(DEV)
        lg = case.logits[torch.from_numpy(np.where(src >= 0, src, -1 - src)).to(DEV)]
    ref = torch.from_numpy((case.old + rng.normal(0, 0.3, T)).astype(np.float32)).to(DEV)

    def run(host):
        dl = torch.empty_like(lg)
        loss, logp, ent = (torch.full((T,), -7.0, device=DEV) for _ in range(3))
        acc = _lib.new_step_acc(DEV)
        terms = dict(kl_kind=_lib.KL_K3, kl_coef=0.1, ref_logp=ref, ent_coef=0.02, entropy_tok=ent)
        if host:
            lh = lg.cpu()
            lh = lh.pin_memory() if pinned else lh
            staging = torch.empty(2 * block * lg.stride(0) * lg.element_size(), dtype=torch.uint8, device=DEV)
            _lib.grpo_logprob_loss_fwd_bwd_host(lh, case.d_target, case.d_old, case.d_adv, case.d_mask, wl.eps,
                                                1.0 / 97, dl, loss, logp, acc, staging, block, tok_src=tok_src,
                                                copy_stream=torch.cuda.Stream() if two_streams else None,
                                                terms=terms)
        else:
            _lib.grpo_logprob_loss_fwd_bwd(lg, case.d_target, case.d_old, case.d_adv, case.d_mask, wl.eps,
                                           1.0 / 97, dl, loss, logp, acc, tok_src=tok_src, terms=terms)
        torch.cuda.synchronize()
        bits = torch.int16 if dtype == "bf16" else torch.int32
        return (dl.view(bits), loss.view(torch.int32), logp.view(torch.int32), ent.view(torch.int32), acc)

    want, got = run(False), run(True)
    for g, w, what in zip(got, want, ("dlogits", "loss", "logp", "entropy", "acc")):
        assert torch.equal(g, w), what
    res = _lib.grpo_finish_step(got[4], got[1].view(torch.float32))
    assert res["status"] == 0 and res["n_valid"] == int(case.mask.sum())


@pytest.mark.parametrize("kind", ["fixed", "dynamic"])
def test_driver_loop_host_logits_equals_device_logits(kind):
    # The driver loop over logits in host memory (each optimizer step streamed through a
    # small staging buffer, copies on their own stream) gives the device loop's bits, with the
    # KL and entropy terms, for fixed chunks and for permuted token-budget bins.
    if kind == "fixed":
        wl = W.make_workload("tiny", rows=8, positions=24, valid_lo=0, V=32776, dtype="bf16", seed=95, std=2.0,
                             mini=4, micro=2)
    else:
        wl = W.make_workload("dynamic", rows=16, len_hi=64, median=20, max_token_len=96, V=32776, seed=96)
    case = H.Case(wl)
    T = wl.T
    ref = torch.from_numpy((case.old + np.random.default_rng(6).normal(0, 0.3, T)).astype(np.float32)).to(DEV)
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    src = np.arange(bp.exec_tokens) if bp.tok_src is None else bp.tok_src
    lg = case.logits[torch.from_numpy(src).to(DEV)]
    ts = None if bp.tok_src is None else torch.from_numpy(bp.tok_src).to(DEV)
    outs = []
    for host in (False, True):
        dl = torch.empty_like(lg)
        loss, logp, ent = (torch.full((T,), -7.0, device=DEV) for _ in range(3))
        accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
        terms = dict(kl_kind=_lib.KL_K3, kl_coef=0.1, ref_logp=ref, ent_coef=0.02, entropy_tok=ent)
        kw = dict(dlogits=dl, target=case.d_target, old_logp=case.d_old, mask=case.d_mask, adv_tok=case.d_adv,
                  loss_tok=loss, logp_tok=logp, accs=accs, clip_eps=wl.eps, tok_src=ts, terms=terms)
        if host:
            block = 13
            staging = torch.empty(2 * block * lg.stride(0) * lg.element_size(), dtype=torch.uint8, device=DEV)
            S.run_batch(bp, logits=None, logits_host=lg.cpu().pin_memory(), staging=staging, block_rows=block,
                        copy_stream=torch.cuda.Stream(), **kw)
        else:
            S.run_batch(bp, logits=lg, side_stream=torch.cuda.Stream(), **kw)
        torch.cuda.synchronize()
        outs.append((dl.view(torch.int16), loss.view(torch.int32), logp.view(torch.int32), ent.view(torch.int32),
                     S.read_results(accs, bp.n_steps)))
    for a, b, what in zip(outs[0], outs[1], ("dlogits", "loss", "logp", "entropy", "results")):
        assert (a == b) if what == "results" else torch.equal(a, b), what


def test_step_captured_in_a_cuda_graph_replays_bitwise():
    # A whole batch (advantage, chunks alternating over two streams, the step finishes) captured
    # once into a CUDA graph: a replay gives the eager run's bits, also after new inputs are
    # written into the same buffers.
    wl = W.make_workload("tiny", rows=8, positions=24, valid_lo=0, V=32776, dtype="bf16", seed=97, std=2.0,
                         mini=4, micro=2)
    case = H.Case(wl)
    T = wl.T
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    rewards, row_tok_off, row_rollout = t(wl.rewards), t(wl.tok_off), t(wl.row_rollout)
    adv_rollout = torch.empty_like(rewards)
    adv_tok = torch.empty(T, device=DEV)
    lg = case.logits.clone()
    dl = torch.empty_like(lg)
    loss, logp = torch.empty(T, device=DEV), torch.empty(T, device=DEV)
    accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()

    def step():
        S.run_batch(bp, logits=lg, dlogits=dl, target=case.d_target, old_logp=case.d_old, mask=case.d_mask,
                    adv_tok=adv_tok, loss_tok=loss, logp_tok=logp, accs=accs, clip_eps=wl.eps, rewards=rewards,
                    adv_rollout=adv_rollout, group_size=wl.group_size, row_tok_off=row_tok_off,
                    row_rollout=row_rollout, side_stream=side)

    def snapshot():
        torch.cuda.synchronize()
        return (dl.view(torch.int16).clone(), loss.clone(), logp.clone(), accs[:].view(-1, _lib.ACC_BYTES)[:, 64:].clone())

    step()  # eager (the first calls also set the kernels' attributes)
    eager = snapshot()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            step()
    for _ in range(2):
        dl.fill_(7.0)
        loss.fill_(7.0)
        g.replay()
        got = snapshot()
        for a, b in zip(got, eager):
            assert torch.equal(a, b)
    # new logits in the same buffer: the replay follows them exactly as an eager run does
    lg.copy_(torch.flip(case.logits, dims=[1]))
    g.replay()
    replayed = snapshot()
    step()
    for a, b in zip(replayed, snapshot()):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[1], eager[1])


def test_all_masked_batch_and_empty_calls_at_product_vocabulary():
    # Degenerate inputs on the product kernels (V = 151936 bf16): a batch with every token
    # masked (no row is read; the producer's scan finds nothing) through the full pass, the
    # forward-only pass and the host-input path, and zero-row calls. Outputs are zeros, the
    # step loss is 0 (not NaN) and N = 0.
    wl = W.make_workload("tiny", rows=4, positions=8, valid_lo=0, V=151936, dtype="bf16", seed=98, std=2.0)
    case = H.Case(wl)
    T = wl.T
    case.mask = np.zeros(T, np.uint8)
    case.d_mask = torch.zeros(T, dtype=torch.uint8, device=DEV)
    for want_grad in (True, False):
        dl, loss, logp, acc = _run_direct(case, 1.0, want_grad=want_grad)
        assert torch.all(loss == 0) and torch.all(logp == 0)
        if want_grad:
            assert torch.all(dl == 0)
        res = _lib.grpo_finish_step(acc, loss, expected_N=0)
        assert res["status"] == 0 and res["n_valid"] == 0 and res["loss"] == 0.0 and res["n_tokens"] == T
    staging = torch.empty(2 * 8 * case.logits.stride(0) * 2, dtype=torch.uint8, device=DEV)
    dl = torch.full_like(case.logits, 3.0)
    loss = torch.full((T,), -7.0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd_host(case.logits.cpu().pin_memory(), case.d_target, case.d_old, case.d_adv,
                                        case.d_mask, 0.2, 1.0, dl, loss, None, acc, staging, 8)
    torch.cuda.synchronize()
    assert torch.all(dl == 0) and torch.all(loss == 0)
    # zero rows: nothing launched, nothing counted
    e = torch.empty((0, 151936), dtype=torch.bfloat16)
    z = torch.empty(0, device=DEV)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd_host(e, torch.empty(0, dtype=torch.int32, device=DEV), None, z,
                                        torch.empty(0, dtype=torch.uint8, device=DEV), 0.2, 1.0, None, z, None, acc,
                                        staging, 8)
    _lib.grpo_logprob_loss_fwd_bwd(e.to(DEV), torch.empty(0, dtype=torch.int32, device=DEV), None, z,
                                   torch.empty(0, dtype=torch.uint8, device=DEV), 0.2, 1.0, None, z, None, acc)
    res = _lib.grpo_finish_step(acc, z, expected_N=0)
    assert res["status"] == 0 and res["n_tokens"] == 0 and res["loss"] == 0.0


def test_row_count_above_int32_is_rejected():
    # a call's rows index the per-token arrays with 32-bit indices: more than 2^31 - 1 rows is
    # an invalid call (checked before anything is read)
    import ctypes
    lib = _lib.lib()
    acc = _lib.new_step_acc(DEV)
    x = torch.zeros((1, 8), device=DEV)
    i = torch.zeros(1, dtype=torch.int32, device=DEV)
    mk = torch.ones(1, dtype=torch.uint8, device=DEV)
    f = torch.zeros(1, device=DEV)
    rc = lib.grpo_logprob_loss_fwd_bwd(x.data_ptr(), _lib.DTYPE_F32, ctypes.c_int64(2 ** 31), 8, 8, None,
                                       i.data_ptr(), None, f.data_ptr(), mk.data_ptr(), ctypes.c_float(0.2),
                                       ctypes.c_float(1.0), None, 0, f.data_ptr(), None, acc.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.ERR_INVALID


@pytest.mark.parametrize("variant", ["c2", "l2"], indirect=True)
def test_extreme_logit_magnitudes(variant):
    # Rows far from the usual scale take the lazy shift's fallback: a row scaled by 30 (a
    # spread of hundreds), rows offset by +300 and by -300. Log-probs are formed without
    # cancellation, so they meet the same bar as ordinary rows; losses and dlogits match the
    # oracle, and the forward-only pass gives the full pass's bits.
    wl = W.make_workload("tiny", rows=4, positions=8, valid_lo=8, V=32776, dtype="bf16", seed=63, std=2.0)
    case = H.Case(wl)
    lg = case.logits.float()
    lg[3] *= 30.0
    lg[9] += 300.0
    lg[17] -= 300.0
    lg = lg.to(torch.bfloat16)
    host = W.logits_to_host(lg)
    scale = 1.0 / 31
    dl, loss, logp, acc = _run_direct(case, scale, logits=lg)
    ref = OL.loss_fwd_bwd(host, wl.target, case.old, case.adv_tok, wl.mask, wl.eps, scale, True)
    gp = H.to_f64(logp)
    assert np.all(np.isfinite(gp))
    assert np.all(np.abs(gp - ref["logp_tok"]) <= 1e-5 * np.maximum(1, np.abs(ref["logp_tok"])))
    got, refd = H.to_f64(dl), ref["dlogits"]
    bad = np.abs(got - refd) > H.dlogits_tol(refd, "bf16")
    bad[H.ambiguous_clip(ref["ratio"], wl.eps)] = False
    assert not bad.any(), np.argwhere(bad)[:3]
    res = _lib.grpo_finish_step(acc, loss)
    assert res["status"] == 0 and res["n_nonfinite"] == 0
    _, loss_f, logp_f, _ = _run_direct(case, scale, want_grad=False, logits=lg)
    assert torch.equal(loss_f, loss) and torch.equal(logp_f, logp)


@pytest.mark.parametrize("variant", ["c2", "l2"], indirect=True)
def test_log_probs_are_shift_invariant(variant):
    # log-softmax is invariant under adding a constant to a row. float32 logits on a 2^-8 grid
    # plus integer shifts are exact, so every shifted row must give the unshifted row's
    # log-probs (up to the arithmetic's own error) and the oracle's, up to the library's stated
    # envelope |LSE| <= 4096; a row shifted past it is reported non-finite.
    V = 32776
    rng = np.random.default_rng(65)
    base = np.round(rng.normal(0, 3.0, V) * 256) / 256
    shifts = [0.0, 100.0, -100.0, 1000.0, -2000.0, 4000.0, 5000.0]
    host = np.stack([base + c for c in shifts]).astype(np.float32)
    assert np.array_equal(host - np.array(shifts, np.float32)[:, None], np.tile(base.astype(np.float32), (7, 1)))
    T = len(shifts)
    lg = torch.from_numpy(host).to(DEV)
    tgt = torch.from_numpy(np.full(T, 123, np.int32)).to(DEV)
    mask = torch.ones(T, dtype=torch.uint8, device=DEV)
    adv = torch.ones(T, device=DEV)
    loss, logp = torch.empty(T, device=DEV), torch.empty(T, device=DEV)
    dl = torch.empty_like(lg)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd(lg, tgt, None, adv, mask, 0.2, 1.0, dl, loss, logp, acc)
    gp = H.to_f64(logp)
    ref = OL.log_softmax_row(base)[123]
    assert np.all(np.abs(gp[:-1] - ref) <= 1e-5 * max(1.0, abs(ref))), (gp, ref)
    assert np.all(np.abs(gp[1:-1] - gp[0]) <= 2e-6 * max(1.0, abs(ref))), gp
    assert not np.isfinite(gp[-1])  # |LSE| above 4096: reported, not returned degraded
    # dlogits (ratio 1, A = 1): p - onehot, the same for every in-range row
    d = H.to_f64(dl)
    p = np.exp(OL.log_softmax_row(base))
    p[123] -= 1.0
    for r in range(T - 1):
        assert np.all(np.abs(d[r] - p) <= 2e-5 * np.abs(p) + 1e-6 * np.abs(p).max()), r


@pytest.mark.parametrize("variant", ["c2", "l2"], indirect=True)
def test_logits_beyond_the_shift_range_are_reported_not_wrong(variant):
    # Rows offset by +-1e30 lie far beyond the envelope |LSE| <= 4096. Their tokens are reported
    # non-finite and the step is skipped with its gradients zeroed: an answer the caller sees,
    # never a silently wrong one. The other rows keep the oracle's log-probs.
    wl = W.make_workload("tiny", rows=4, positions=8, valid_lo=8, V=32776, dtype="bf16", seed=64, std=2.0)
    case = H.Case(wl)
    lg = case.logits.float()
    lg[9] += 1e30
    lg[17] -= 1e30
    lg = lg.to(torch.bfloat16)
    host = W.logits_to_host(lg)
    dl, loss, logp, acc = _run_direct(case, 1.0 / 31, logits=lg)
    gp = H.to_f64(logp)
    assert not np.isfinite(gp[9]) and not np.isfinite(gp[17])
    ok = np.ones(wl.T, bool)
    ok[[9, 17]] = False
    ref = OL.loss_fwd_bwd(host[ok], wl.target[ok], case.old[ok], case.adv_tok[ok], wl.mask[ok], wl.eps,
                          1.0 / 31, False)
    assert np.all(np.abs(gp[ok] - ref["logp_tok"]) <= 1e-5 * np.maximum(1, np.abs(ref["logp_tok"])))
    res = _lib.grpo_finish_step(acc, loss, grad_bufs=[dl])
    assert res["status"] == _lib.STEP_SKIPPED_NONFINITE and res["n_nonfinite"] == 2
    assert torch.all(dl == 0)


@pytest.mark.parametrize("world", [2, 3])
def test_data_parallel_row_blocks_match_the_whole_step(world):
    # The row blocks data-parallel ranks would run, run one after another on this GPU: each
    # with the step's global scale 1/N and a finish whose divisor is N. Per-token outputs and
    # dlogits are the whole step's bits; the combined step result is the whole step's (the
    # float64 loss sum up to the order of its additions).
    wl = W.make_workload("qwen_step", rows=8, len_lo=20, len_hi=40, seed=77, mini=8, micro=8)
    case = H.Case(wl)
    T = case.logits.shape[0]
    N = int(wl.mask.sum())
    dl, loss, logp, acc = _run_direct(case, 1.0 / N)
    whole = _lib.grpo_finish_step(acc, loss, expected_N=N)
    dl_s = torch.full_like(case.logits, 7.0)
    loss_s = torch.full((T,), -7.0, device=DEV)
    logp_s = torch.full((T,), -7.0, device=DEV)
    parts = []
    for r in range(world):
        lo, hi = S.dp_row_block(8, r, world)
        t0, t1 = int(wl.tok_off[lo]), int(wl.tok_off[hi])
        a = _lib.new_step_acc(DEV)
        _lib.grpo_logprob_loss_fwd_bwd(case.logits[t0:t1], case.d_target[t0:t1], case.d_old[t0:t1],
                                       case.d_adv[t0:t1], case.d_mask[t0:t1], wl.eps, 1.0 / N, dl_s[t0:t1],
                                       loss_s[t0:t1], logp_s[t0:t1], a)
        parts.append(_lib.grpo_finish_step_ex(a, loss_s[t0:t1], divisor=N,
                                              expected_N=int(wl.mask[t0:t1].sum())))
    torch.cuda.synchronize()
    assert torch.equal(dl_s.view(torch.int16), dl.view(torch.int16))
    assert torch.equal(loss_s.view(torch.int32), loss.view(torch.int32))
    assert torch.equal(logp_s.view(torch.int32), logp.view(torch.int32))
    got = S.combine_step_results(parts, N)
    for k in ("n_valid", "n_clipped", "n_nonfinite", "n_tokens", "status", "kernel_flags"):
        assert got[k] == whole[k], k
    assert got["clipfrac"] == whole["clipfrac"]
    bound = 1e-12 * float(torch.abs(loss.double()).sum()) / N
    assert abs(got["loss"] - whole["loss"]) <= bound
    assert all(p["loss"] == p["loss_sum"] / N for p in parts)
